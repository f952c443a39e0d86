// k_softmax.cu -- masked row softmax over the band and its backward.
//
// Forward (nvFuser issue "HuggingFace BertForMaskedLM - Log Softmax Fusion
// with Autocast has bad perf", fusion 1: row max, exp of the difference, row
// sum, division, all in fp32):
//     P[i,t] = exp(S[i,t] - m_i) / Z_i   on the valid slots t in
//              [t_lo(i), t_hi(i)], 0 elsewhere;  lse_i = m_i + log Z_i,
// with the valid range in closed form: t_lo = max(0, w - floor(i/s)),
// t_hi = min(D-1, w + floor((n-1-i)/s)).
// Backward:  dS = P * (dP - delta_i), delta_i = sum over valid slots P*dP.
//
// One warp per band row.  A band row of D elements starts at an arbitrary
// element boundary, so the warp walks the row's aligned 16-byte pieces
// (128-bit loads, 32 consecutive pieces per warp instruction).  Pieces that
// straddle a row boundary are shared with the neighbouring row's warp: they
// are read whole but written element by element, only the elements of this
// row; every other piece is written with one 128-bit store.  Two passes: the
// reduction, then the write; the second pass re-reads the row from L1/L2.
#include "swab_internal.h"

namespace swab {
namespace {

constexpr int kRowsPerBlock = 8;  // warps per CTA

template <typename T> struct Vec {
    static constexpr int N = 16 / sizeof(T);  // elements per 16-byte piece
};

template <typename T>
__device__ __forceinline__ void unpack(const uint4 &v, float (&x)[Vec<T>::N]) {
    if constexpr (sizeof(T) == 4) {
        x[0] = __uint_as_float(v.x);
        x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z);
        x[3] = __uint_as_float(v.w);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = lo16<T>(w[k]);
            x[2 * k + 1] = hi16<T>(w[k]);
        }
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack(const float (&x)[Vec<T>::N]) {
    if constexpr (sizeof(T) == 4) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                          __float_as_uint(x[3]));
    } else {
        return make_uint4(pack2<T>(x[0], x[1]), pack2<T>(x[2], x[3]), pack2<T>(x[4], x[5]),
                          pack2<T>(x[6], x[7]));
    }
}

struct RowSpan {
    long long e0;       // first element of the row
    long long c0, c1;   // first / last aligned piece touching the row
    int t_lo, t_hi;     // valid slots
};

__device__ __forceinline__ RowSpan row_span(const Geom &g, long long R, int epc) {
    RowSpan rs;
    const int i = (int)(R % g.n);
    rs.e0 = R * g.D;
    rs.c0 = rs.e0 / epc;
    rs.c1 = (rs.e0 + g.D - 1) / epc;
    rs.t_lo = max(0, g.w - i / g.s);
    rs.t_hi = min(g.D - 1, g.w + (g.n - 1 - i) / g.s);
    return rs;
}

template <typename T>
__device__ __forceinline__ void store_piece(T *base, long long piece, const RowSpan &rs,
                                            int D, const float (&y)[Vec<T>::N]) {
    constexpr int N = Vec<T>::N;
    const long long pe = piece * N;
    if (pe >= rs.e0 && pe + N <= rs.e0 + D) {
        *reinterpret_cast<uint4 *>(base + pe) = pack<T>(y);
    } else {
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const long long e = pe + u;
            if (e >= rs.e0 && e < rs.e0 + D) base[e] = Elt<T>::from_f(y[u]);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_band_softmax_stream(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const long long R = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (R >= (long long)g.BH * g.n) return;
    const RowSpan rs = row_span(g, R, N);
    const T *S = reinterpret_cast<const T *>(p.S);
    // pass 1: running max / sum of this lane's valid elements
    float m = -INFINITY, z = 0.f;
    for (long long c = rs.c0 + lane; c <= rs.c1; c += 32) {
        float x[N];
        unpack<T>(ldg16(S + c * N), x);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const long long t = c * N + u - rs.e0;
            if (t >= rs.t_lo && t <= rs.t_hi) {
                if (x[u] > m) {
                    z = z * expf(m - x[u]) + 1.f;
                    m = x[u];
                } else {
                    z += expf(x[u] - m);
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
        const float mn = fmaxf(m, m2);
        z = (m == -INFINITY ? 0.f : z * expf(m - mn)) + (m2 == -INFINITY ? 0.f : z2 * expf(m2 - mn));
        m = mn;
    }
    const float inv = 1.f / z;
    // pass 2: probabilities
    T *P = reinterpret_cast<T *>(p.P);
    for (long long c = rs.c0 + lane; c <= rs.c1; c += 32) {
        float x[N];
        unpack<T>(ldg16(S + c * N), x);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const long long t = c * N + u - rs.e0;
            x[u] = (t >= rs.t_lo && t <= rs.t_hi) ? expf(x[u] - m) * inv : 0.f;
        }
        store_piece<T>(P, c, rs, g.D, x);
    }
    if (p.lse && lane == 0) p.lse[R] = m + logf(z);
}

template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_band_softmax_bwd_stream(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const long long R = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (R >= (long long)g.BH * g.n) return;
    const RowSpan rs = row_span(g, R, N);
    const T *P = reinterpret_cast<const T *>(p.S);
    const T *dP = reinterpret_cast<const T *>(p.S2);
    float delta = 0.f;
    for (long long c = rs.c0 + lane; c <= rs.c1; c += 32) {
        float x[N], y[N];
        unpack<T>(ldg16(P + c * N), x);
        unpack<T>(ldg16(dP + c * N), y);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const long long t = c * N + u - rs.e0;
            if (t >= rs.t_lo && t <= rs.t_hi) delta = fmaf(x[u], y[u], delta);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
    T *dS = reinterpret_cast<T *>(p.P);
    for (long long c = rs.c0 + lane; c <= rs.c1; c += 32) {
        float x[N], y[N];
        unpack<T>(ldg16(P + c * N), x);
        unpack<T>(ldg16(dP + c * N), y);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const long long t = c * N + u - rs.e0;
            x[u] = (t >= rs.t_lo && t <= rs.t_hi) ? x[u] * (y[u] - delta) : 0.f;
        }
        store_piece<T>(dS, c, rs, g.D, x);
    }
}

// Register-resident variants: the row's pieces (at most NCH per lane) are
// read once and kept in registers.
template <typename T, int NCH>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_band_softmax_reg(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    constexpr bool kKeep = NCH * N <= 32;  // keep exp() values, else recompute
    constexpr float kLog2e = 1.4426950408889634f;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const long long R = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (R >= (long long)g.BH * g.n) return;
    const RowSpan rs = row_span(g, R, N);
    const T *S = reinterpret_cast<const T *>(p.S);
    uint4 raw[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const long long c = rs.c0 + lane + 32 * k;
        raw[k] = c <= rs.c1 ? ldg16(S + c * N) : make_uint4(0, 0, 0, 0);
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N];
        unpack<T>(raw[k], x);
        const long long t0 = (rs.c0 + lane + 32 * k) * N - rs.e0;
#pragma unroll
        for (int u = 0; u < N; ++u)
            if (t0 + u >= rs.t_lo && t0 + u <= rs.t_hi) m = fmaxf(m, x[u]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float mb = m * kLog2e;
    float z = 0.f;
    float e[kKeep ? NCH * N : 1];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N];
        unpack<T>(raw[k], x);
        const long long t0 = (rs.c0 + lane + 32 * k) * N - rs.e0;
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const bool v = t0 + u >= rs.t_lo && t0 + u <= rs.t_hi;
            const float ev = v ? exp2f(fmaf(x[u], kLog2e, -mb)) : 0.f;
            z += ev;
            if constexpr (kKeep) e[k * N + u] = ev;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float inv = 1.f / z;
    T *P = reinterpret_cast<T *>(p.P);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const long long c = rs.c0 + lane + 32 * k;
        if (c > rs.c1) break;
        float y[N];
        if constexpr (kKeep) {
#pragma unroll
            for (int u = 0; u < N; ++u) y[u] = e[k * N + u] * inv;
        } else {
            float x[N];
            unpack<T>(raw[k], x);
            const long long t0 = c * N - rs.e0;
#pragma unroll
            for (int u = 0; u < N; ++u) {
                const bool v = t0 + u >= rs.t_lo && t0 + u <= rs.t_hi;
                y[u] = v ? exp2f(fmaf(x[u], kLog2e, -mb)) * inv : 0.f;
            }
        }
        store_piece<T>(P, c, rs, g.D, y);
    }
    if (p.lse && lane == 0) p.lse[R] = m + logf(z);
}

template <typename T, int NCH>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_band_softmax_bwd_reg(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const long long R = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (R >= (long long)g.BH * g.n) return;
    const RowSpan rs = row_span(g, R, N);
    const T *P = reinterpret_cast<const T *>(p.S);
    const T *dP = reinterpret_cast<const T *>(p.S2);
    uint4 rp[NCH], rd[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const long long c = rs.c0 + lane + 32 * k;
        rp[k] = c <= rs.c1 ? ldg16(P + c * N) : make_uint4(0, 0, 0, 0);
        rd[k] = c <= rs.c1 ? ldg16(dP + c * N) : make_uint4(0, 0, 0, 0);
    }
    float delta = 0.f;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N], y[N];
        unpack<T>(rp[k], x);
        unpack<T>(rd[k], y);
        const long long t0 = (rs.c0 + lane + 32 * k) * N - rs.e0;
#pragma unroll
        for (int u = 0; u < N; ++u)
            if (t0 + u >= rs.t_lo && t0 + u <= rs.t_hi) delta = fmaf(x[u], y[u], delta);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
    T *dS = reinterpret_cast<T *>(p.P);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const long long c = rs.c0 + lane + 32 * k;
        if (c > rs.c1) break;
        float x[N], y[N];
        unpack<T>(rp[k], x);
        unpack<T>(rd[k], y);
        const long long t0 = c * N - rs.e0;
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const bool v = t0 + u >= rs.t_lo && t0 + u <= rs.t_hi;
            x[u] = v ? x[u] * (y[u] - delta) : 0.f;
        }
        store_piece<T>(dS, c, rs, g.D, x);
    }
}

template <typename T>
cudaError_t launch_sm(const SoftmaxArgs &a, bool bwd, cudaStream_t st) {
    constexpr int N = Vec<T>::N;
    const long long rows = (long long)a.g.BH * a.g.n;
    const unsigned blocks = (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    const dim3 blk(kRowsPerBlock * 32);
    // most aligned pieces a row can touch, spread over 32 lanes
    const long long pieces = (a.g.D + N - 1) / N + 1;
    const long long per_lane = (pieces + 31) / 32;
    if (bwd) {
        if (per_lane <= 1) k_band_softmax_bwd_reg<T, 1><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 2) k_band_softmax_bwd_reg<T, 2><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 3) k_band_softmax_bwd_reg<T, 3><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 4) k_band_softmax_bwd_reg<T, 4><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 8) k_band_softmax_bwd_reg<T, 8><<<blocks, blk, 0, st>>>(a);
        else k_band_softmax_bwd_stream<T><<<blocks, blk, 0, st>>>(a);
    } else {
        if (per_lane <= 1) k_band_softmax_reg<T, 1><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 2) k_band_softmax_reg<T, 2><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 3) k_band_softmax_reg<T, 3><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 4) k_band_softmax_reg<T, 4><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 8) k_band_softmax_reg<T, 8><<<blocks, blk, 0, st>>>(a);
        else if (per_lane <= 17) k_band_softmax_reg<T, 17><<<blocks, blk, 0, st>>>(a);
        else k_band_softmax_stream<T><<<blocks, blk, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band_softmax(DType dt, const SoftmaxArgs &a, cudaStream_t st) {
    if (dt == kF32) return launch_sm<float>(a, false, st);
    if (dt == kF16) return launch_sm<__half>(a, false, st);
    return launch_sm<__nv_bfloat16>(a, false, st);
}

cudaError_t launch_band_softmax_bwd(DType dt, const SoftmaxArgs &a, cudaStream_t st) {
    if (dt == kF32) return launch_sm<float>(a, true, st);
    if (dt == kF16) return launch_sm<__half>(a, true, st);
    return launch_sm<__nv_bfloat16>(a, true, st);
}

}  // namespace swab
