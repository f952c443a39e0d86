// k_bias_transpose.cu -- AddBiasTranspose: the bias add and the
// [b, n, M, h, hd] -> [M, b, h, n, hd] transpose after the merged projection in
// one pass (ONNX Runtime issue "[WIP] Improve LongformerAttention
// performance", item (2); conclusion (g): the widest vector accesses win).
//
// One thread per 16-byte chunk of a row of X, in X's order, so every warp
// reads 512 contiguous bytes; the chunk's destination row segment (hd elements
// of one (m, b, h, i)) is contiguous in Y, so the writes come in whole
// 128-byte lines for hd = 64 half.  Each thread keeps four rows' loads in
// flight before its stores.  The sum is formed in fp32 and rounded once: fp32 holds
// at least 2p + 2 bits for p-bit fp16 / bf16 significands, so the double
// rounding is innocuous and the result is the correctly rounded sum.
// HBM-bound: 2 * b*n*M*h*hd * size bytes (plus the bias, L2-resident).
#include "swab_internal.h"

static constexpr unsigned kSwabFile = 5;   // site id of the bounds checks

namespace swab {
namespace {

template <typename T>
__device__ __forceinline__ uint4 add_chunk(const uint4 &x, const uint4 &b) {
    if constexpr (sizeof(T) == 4) {
        return make_uint4(__float_as_uint(__uint_as_float(x.x) + __uint_as_float(b.x)),
                          __float_as_uint(__uint_as_float(x.y) + __uint_as_float(b.y)),
                          __float_as_uint(__uint_as_float(x.z) + __uint_as_float(b.z)),
                          __float_as_uint(__uint_as_float(x.w) + __uint_as_float(b.w)));
    } else {
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, bw[4] = {b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = pack2<T>(lo16<T>(xw[k]) + lo16<T>(bw[k]), hi16<T>(xw[k]) + hi16<T>(bw[k]));
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}

constexpr int kRowsPerThread = 4;   // rows of X per thread: loads in flight before the stores

// Thread x of block (bx, by) owns chunk q = bx * blockDim + x of every row of X
// (a row holds M * h * cpr chunks) and rows by * kRowsPerThread .. + 3 (then
// every gridDim.y * kRowsPerThread rows).  Its
// (m, hh, cc) -- and so its bias chunk and its place in Y -- are fixed.
template <typename T>
__global__ void __launch_bounds__(256) k_add_bias_transpose(const BiasTransposeArgs p) {
    const unsigned chunks_per_row = (unsigned)(p.M * p.h * p.cpr);
    const unsigned q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= chunks_per_row) return;
    const unsigned cc = q % (unsigned)p.cpr, mh = q / (unsigned)p.cpr;
    const unsigned hh = mh % (unsigned)p.h, m = mh / (unsigned)p.h;
    uint4 bv = make_uint4(0, 0, 0, 0);
    if (p.bias) bv = ldg16(GP(p.bnd, reinterpret_cast<const uint4 *>(p.bias) + q));   // bias is [M, h, cpr]
    // Y chunk of (m, bb, hh, i, cc): ((m * b + bb) * h + hh) * n + i, times cpr, plus cc
    const long long ybase = (((long long)m * p.b * p.h + hh) * p.n) * p.cpr + cc;
    const uint4 *X = reinterpret_cast<const uint4 *>(p.X);
    uint4 *Y = reinterpret_cast<uint4 *>(p.Y);
    for (long long row0 = (long long)blockIdx.y * kRowsPerThread; row0 < p.rows;
         row0 += (long long)gridDim.y * kRowsPerThread) {
        uint4 v[kRowsPerThread];
#pragma unroll
        for (int k = 0; k < kRowsPerThread; ++k) {
            const long long row = row0 + k;
            v[k] = row < p.rows ? ldg16(GP(p.bnd, X + row * chunks_per_row + q)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kRowsPerThread; ++k) {
            const long long row = row0 + k;   // below 2^31 (checked by the caller)
            if (row >= p.rows) break;
            const unsigned bb = (unsigned)row / (unsigned)p.n, i = (unsigned)row - bb * (unsigned)p.n;
            const uint4 y = p.bias ? add_chunk<T>(v[k], bv) : v[k];
            *GP(p.bnd, Y + ybase + ((long long)bb * p.h * p.n + i) * p.cpr) = y;
        }
    }
}

}  // namespace

cudaError_t launch_add_bias_transpose(DType dt, const BiasTransposeArgs &a, cudaStream_t st) {
    const long long per_row = a.M * a.h * a.cpr;
    if (per_row == 0 || a.rows == 0) return cudaSuccess;
    if (per_row > (1LL << 30) || a.rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    const long long ry = (a.rows + kRowsPerThread - 1) / kRowsPerThread;
    const unsigned threads = 256;
    const dim3 grid((unsigned)((per_row + threads - 1) / threads), (unsigned)(ry < 65535 ? ry : 65535));
    if (dt == kF32) k_add_bias_transpose<float><<<grid, threads, 0, st>>>(a);
    else if (dt == kF16) k_add_bias_transpose<__half><<<grid, threads, 0, st>>>(a);
    else k_add_bias_transpose<__nv_bfloat16><<<grid, threads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace swab
