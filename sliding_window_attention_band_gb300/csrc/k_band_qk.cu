// k_band_qk.cu -- the forward banded product ("Developing a faster schedule
// for Longformer's kernel", TVM forum, post 6: dense x dense^T restricted to
// t3d3 = w + w_upper + 1 diagonals):
//     S[i,t] = alpha * A[i] . B[i + (t-w)*s]   (padding where the key is
//     outside the sequence).
//
// Tensor-core kernel (f16 / bf16, head_dim 64).  One CTA owns 128 query rows
// of one residue r (rows r + s*a, a in [a0, a0+128)) and one 128-key chunk of
// the keys its band touches.  The product is one dense 128x128x64 tcgen05.mma
// into tensor memory with the KEY chunk as the M operand (TMEM lane = key,
// column = query); out-of-band entries are simply not stored.  For a fixed
// query the 32 lanes of a warp hold 32 consecutive band slots of that
// query's row, so each store instruction writes 64 contiguous bytes; each
// lane works out once per chunk which queries its key belongs to and where
// the first of them goes, so a store costs a compare and a pointer step.
// (A query-major epilogue -- TMEM lane = query, each thread streaming its
// own band row in aligned 32-byte pieces -- was 35.5 us against 31.9 us at
// n = 4096, w = 256, and 920 against 801 us at n = 32768, w = 4096.)
//
// Warp roles (192 threads): warp 0 issues TMA loads (query tile once, key
// chunks into a 2-stage ring), warp 1 owns tensor memory and issues the MMA
// into one 128-column accumulator, warps 2-5 drain it.  The CTA is kept small
// (50 KB of shared memory, 128 TMEM columns, at most 96 registers a thread)
// so that three CTAs share an SM: one CTA's MMA and loads run while another
// drains.
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 3;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kBM = 128;          // keys per chunk (MMA M)
constexpr int kBN = 128;          // queries per tile (MMA N)
constexpr int kStages = 2;        // key-chunk ring depth
// A query tile's key chunks write disjoint band slots: one CTA per chunk
// balances the SMs best.
constexpr int kThreads = 192;
constexpr int kTileBytes = 128 * 128;  // 128 rows x 64 halves
constexpr int kSmemBytes = kStages * kTileBytes + kTileBytes + 1024 /*barriers*/ + 1024 /*align*/;
constexpr uint32_t kTmemCols = 128;   // one 128 x 128 fp32 accumulator

template <typename T>
__global__ void __launch_bounds__(kThreads, 3)
    k_band_qk_tc(const __grid_constant__ TmapSet mapA, const __grid_constant__ TmapSet mapB,
                 const QKArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ktile = base;                                 // kStages x 16 KB (A: keys)
    uint8_t *qtile = base + kStages * kTileBytes;          // 16 KB (B: queries)
    uint64_t *bars = reinterpret_cast<uint64_t *>(qtile + kTileBytes);
    uint64_t *kfull = bars;                 // [kStages]
    uint64_t *kempty = bars + kStages;      // [kStages]
    uint64_t *qfull = bars + 2 * kStages;   // [1]
    uint64_t *tfull = qfull + 1;            // [2]
    uint64_t *tempty = tfull + 2;           // [2]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, bh = blockIdx.z;
    const int nr = residue_len(g.n, g.s, r);
    const int nsplit = p.nsplit > 0 ? p.nsplit : 1;   // chunks of a query tile, a CTA each
    const int split = blockIdx.x % nsplit;
    const int a0 = (blockIdx.x / nsplit) * kBN;
    if (a0 >= nr) return;  // whole CTA leaves before any barrier or allocation
    const int kb_tile = max(a0 - g.w, 0);   // the tile's first key
    const int kb_hi = min(a0 + kBN - 1 + g.wu, nr - 1);
    const int nck_tile = (kb_hi - kb_tile + kBM) / kBM;
    const int c_first = split;
    if (c_first >= nck_tile) return;
    // this CTA's chunk: c_first of the tile
    const int kb_lo = kb_tile + c_first * kBM;
    const int nck = 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
        }
        mbar_init(qfull, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 128);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap *ma = &mapA.m[r];
            const CUtensorMap *mb = &mapB.m[r];
            tma_prefetch_desc(ma);
            tma_prefetch_desc(mb);
            mbar_arrive_expect_tx(qfull, kTileBytes);
            tma_load_3d(qtile, ma, qfull, 0, a0, bh);
            for (int c = 0; c < nck; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                if (!mbar_wait(&kempty[st], ph ^ 1, abort_flag, p.err)) break;
                mbar_arrive_expect_tx(&kfull[st], kTileBytes);
                tma_load_3d(ktile + st * kTileBytes, mb, &kfull[st], 0, kb_lo + c * kBM, bh);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr bool kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
            const uint32_t idesc = idesc_f16(kBM, kBN, kBf16, false, false);
            const uint32_t q_addr = smem_u32(qtile);
            if (mbar_wait(qfull, 0, abort_flag, p.err)) {
                for (int c = 0; c < nck; ++c) {
                    const int st = c % kStages;
                    const uint32_t ph = (c / kStages) & 1;
                    const int b = 0;
                    const uint32_t bph = c & 1;
                    if (!mbar_wait(&kfull[st], ph, abort_flag, p.err)) break;
                    if (!mbar_wait(&tempty[b], bph ^ 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(ktile + st * kTileBytes);
                    const uint32_t d = tmem + b * kBN;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t kd = sdesc_sw128(k_addr + 32 * k, 16, 1024);
                        const uint64_t qd = sdesc_sw128(q_addr + 32 * k, 16, 1024);
                        mma_f16_ss(d, kd, qd, idesc, k > 0);
                    }
                    mma_commit(&kempty[st]);
                    mma_commit(&tfull[b]);
                }
            }
        }
    } else {
        // epilogue: warps 2..5, TMEM lane quarter = warp % 4
        const int quarter = warp & 3;
        T *S = reinterpret_cast<T *>(p.S);
        const int m = quarter * 32 + lane;  // key within the chunk
        const long long row0 = (long long)bh * g.n + r + (long long)g.s * a0;
        const long long stepq = (long long)g.s * g.D - 1;  // offset change per query
        const float alpha = p.alpha;
        for (int c = 0; c < nck; ++c) {
            const int b = 0;
            const uint32_t bph = c & 1;
            const bool ok = mbar_wait(&tfull[b], bph, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, ok)) break;  // keep the warp converged for tcgen05.ld
            tc_fence_after();
            const int kk = kb_lo + c * kBM + m;  // key sub-index of this lane
            const int tq0 = kk - a0 + g.w;  // slot of query a0; query q has tq0 - q
            // the queries whose band holds this key: slot tq0 - q in [0, D),
            // query inside its residue; none for a key past the band's end
            const int qlo = max(tq0 - g.D + 1, 0);
            const int qhi = kk <= kb_hi ? min(tq0, nr - 1 - a0) : -1;
            // element (query a0, this key); query q is q*stepq further
            T *const col = S + row0 * g.D + tq0;
#pragma unroll 1
            for (int grp = 0; grp < 4; ++grp) {
                // the group's queries [32 grp, +32): none of them in any lane's
                // range (an edge chunk) -- skip; all of them in every lane's
                // range (the band's interior) -- store without a compare
                const int g0 = grp * 32;
                if (!__any_sync(0xffffffffu, qlo <= g0 + 31 && qhi >= g0)) continue;
                const bool all_in = __all_sync(0xffffffffu, qlo <= g0 && qhi >= g0 + 31);
                uint32_t v[32];
                tmem_ld32(tmem_addr(tmem, quarter * 32, b * kBN + g0), v);
                tmem_ld_wait();
                T *dst = col + (long long)g0 * stepq;
                if (all_in) {
#pragma unroll
                    for (int j = 0; j < 32; ++j, dst += stepq) *GP(g.bnd, dst) = Elt<T>::from_f(alpha * __uint_as_float(v[j]));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j, dst += stepq) {
                        const int q = g0 + j;
                        if (q >= qlo && q <= qhi) *GP(g.bnd, dst) = Elt<T>::from_f(alpha * __uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[b]);
        }
        // padding: slots whose key lies outside [0, nr) (the tile's first CTA)
        const T pad = Elt<T>::from_f(g.padding);
        for (int q = warp - 2; split == 0 && q < kBN; q += 4) {
            const int qq = a0 + q;
            if (qq >= nr) break;
            const int t_lo = max(0, g.w - qq);
            const int t_hi = min(g.D - 1, g.w + nr - 1 - qq);
            T *row = S + ((long long)bh * g.n + r + (long long)g.s * qq) * g.D;
            for (int t = lane; t < t_lo; t += 32) *GP(g.bnd, row + t) = pad;
            for (int t = t_hi + 1 + lane; t < g.D; t += 32) *GP(g.bnd, row + t) = pad;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// exact fp32 path: one CTA per query row, threads over slots, FFMA dot products
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_band_qk_f32(const DenseArgs p) {
    const Geom &g = p.g;
    const long long R = blockIdx.x;  // row in [0, BH*n)
    const int i = (int)(R % g.n);
    const long long bh = R / g.n;
    __shared__ float arow[128];
    const float *A = reinterpret_cast<const float *>(p.A) + R * g.hd;
    const float *B = reinterpret_cast<const float *>(p.B) + bh * g.n * g.hd;
    for (int c = threadIdx.x; c < g.hd; c += blockDim.x) arow[c] = *GP(g.bnd, A + c);
    __syncthreads();
    float *S = reinterpret_cast<float *>(p.out) + R * g.D;
    for (int t = threadIdx.x; t < g.D; t += blockDim.x) {
        const long long j = (long long)i + (long long)(t - g.w) * g.s;
        if (j < 0 || j >= g.n) {
            *GP(g.bnd, S + t) = g.padding;
        } else {
            const float *b = B + j * g.hd;
            float acc = 0.f;
            for (int c = 0; c < g.hd; ++c) acc = fmaf(arow[c], *GP(g.bnd, b + c), acc);
            *GP(g.bnd, S + t) = p.alpha * acc;
        }
    }
}

template <typename T>
cudaError_t launch_qk(const TmapSet &mapA, const TmapSet &mapB, const QKArgs &a0, cudaStream_t st) {
    const int tiles = (a0.g.nsub + kBN - 1) / kBN;
    // key chunks of a tile at most: its band spans kBN - 1 + w + w_upper keys
    const long long max_nck = ((long long)kBN - 1 + a0.g.w + a0.g.wu + kBM) / kBM + 1;
    QKArgs a = a0;
    a.nsplit = (int)max_nck;   // a CTA per chunk
    if ((long long)tiles * a.nsplit > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)(tiles * a.nsplit), a.g.s, a.g.BH);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_band_qk_tc<T>), kSmemBytes);
    if (e != cudaSuccess) return e;
    k_band_qk_tc<T><<<grid, kThreads, kSmemBytes, st>>>(mapA, mapB, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band_qk_tc(DType dt, const TmapSet &mapA, const TmapSet &mapB,
                              const QKArgs &a, cudaStream_t st) {
    return dt == kF16 ? launch_qk<__half>(mapA, mapB, a, st) : launch_qk<__nv_bfloat16>(mapA, mapB, a, st);
}

cudaError_t launch_band_qk_f32(const DenseArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    k_band_qk_f32<<<(unsigned)rows, 128, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace swab
