// k_band_qk.cu -- the forward banded product ("Developing a faster schedule
// for Longformer's kernel", TVM forum, post 6: dense x dense^T restricted to
// t3d3 = w + w_upper + 1 diagonals):
//     S[i,t] = alpha * A[i] . B[i + (t-w)*s]   (padding where the key is
//     outside the sequence).
//
// Tensor-core kernel (f16 / bf16, head_dim 64).  One CTA owns 128 query rows
// of one residue r (rows r + s*a, a in [a0, a0+128)) and walks the keys its
// band touches, 128 at a time.  Each step is one dense 128x128x64 product
// computed with tcgen05.mma into tensor memory.  Out-of-band entries of the
// dense tile are simply not stored.  Two epilogues:
//
//  * ROWS (used when s*D - 1 is a multiple of 16, e.g. every undilated band
//    with D = 2^k + 1): the QUERY tile is the M operand, so TMEM lane = query
//    row and each thread streams its own band row.  Consecutive chunks hand a
//    row consecutive slots, and because the row pitch minus one is a
//    multiple of 16 elements, every row of the CTA has the same offset modulo
//    32 bytes.  The epilogue is compiled once per offset (16 cases, picked
//    once per CTA): each 32-value TMEM group becomes two aligned 32-byte
//    pieces (one st.global.v8 each, a full sector), carrying the leftover
//    values in registers to the next group or chunk.  Only the two pieces at
//    the ends of a row's valid range are stored element by element.
//  * KEYS (any geometry): the KEY chunk is the M operand, TMEM lane = key,
//    column = query; for a fixed query the 32 lanes of a warp hold 32
//    consecutive band slots of that query's row, so each store instruction
//    writes 64 contiguous bytes.
//
// Warp roles (192 threads): warp 0 issues TMA loads (query tile once, key
// chunks into a 2-stage ring), warp 1 owns tensor memory and issues the MMAs
// into one 128-column accumulator, warps 2-5 drain it.  The CTA is kept small
// (50 KB of shared memory, 128 TMEM columns, at most 96 registers a thread)
// so that three CTAs share an SM: one CTA's MMA and loads run while another
// drains, and 384 tiles of the n = 4096 band fit in one wave.  (Two CTAs an
// SM with a 4-stage ring and two accumulators: 45.8 / 72.4 us at dilation
// 0 / 3 against 35.5 / 49.8 us.)
#include <type_traits>

#include "swab_internal.h"

namespace swab {
namespace {

constexpr int kBM = 128;          // keys per chunk (MMA M)
constexpr int kBN = 128;          // queries per tile (MMA N)
constexpr int kStages = 2;        // key-chunk ring depth
// A query tile's key chunks write disjoint band slots, so they can be split
// over CTAs.  With the KEYS epilogue a CTA per chunk balances the SMs best
// (49.8 -> 45.7 us at n = 4096, w = 256, dilation 3); the ROWS epilogue
// keeps whole tiles (a split costs it a Q load and two partly shared pieces
// a row a chunk: 35.5 -> 42 us).
template <bool kRows> __host__ __device__ constexpr int chunks_per_cta() { return kRows ? (1 << 20) : 1; }
constexpr int kThreads = 192;
constexpr int kTileBytes = 128 * 128;  // 128 rows x 64 halves
constexpr int kSmemBytes = kStages * kTileBytes + kTileBytes + 1024 /*barriers*/ + 1024 /*align*/;
constexpr uint32_t kTmemCols = 128;   // one 128 x 128 fp32 accumulator

__device__ __forceinline__ void stg_v8(void *ptr, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Store 16 consecutive values (elements 16*P .. 16*P+15 of `base`, a 32-byte
// aligned pointer); elements outside [lo, hi] are left untouched.
template <typename T>
__device__ __forceinline__ void store_piece16(T *base, long long P, const float (&y)[16],
                                              long long lo, long long hi) {
    const long long e0 = P * 16;
    if (e0 >= lo && e0 + 15 <= hi) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = pack2<T>(y[2 * k], y[2 * k + 1]);
        stg_v8(base + e0, w);
    } else if (e0 + 15 >= lo && e0 <= hi) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (e0 + u >= lo && e0 + u <= hi) base[e0 + u] = Elt<T>::from_f(y[u]);
    }
}

struct RowsCtx {
    uint64_t *tfull, *tempty;
    volatile int *abort_flag;
    unsigned *err;
    uint32_t lane_base;  // TMEM address of this warp's lane quarter, column 0
    int nck;
    long long piece0;    // piece of value 0 of chunk 0 (its first DL positions precede it)
    long long ev_lo, ev_hi;  // valid elements of this thread's row
    float alpha;
};

// ROWS epilogue for one thread = one query row; DL = offset of the row's
// chunk-0 value 0 inside its 16-element piece.
template <typename T, int DL>
__device__ __noinline__ void qk_rows_epilogue(const RowsCtx &x, T *base) {
    float carry[DL > 0 ? DL : 1];
#pragma unroll
    for (int i = 0; i < (DL > 0 ? DL : 1); ++i) carry[i] = 0.f;
    for (int c = 0; c < x.nck; ++c) {
        const int b = 0;
        const uint32_t bph = c & 1;
        const bool ok = mbar_wait(&x.tfull[b], bph, x.abort_flag, x.err);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
#pragma unroll 1
        for (int grp = 0; grp < 4; ++grp) {
            uint32_t v[32];
            tmem_ld32(x.lane_base + b * kBN + grp * 32, v);
            tmem_ld_wait();
            float y[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = x.alpha * __uint_as_float(v[i]);
            float pa[16], pb[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                if constexpr (DL > 0) pa[q] = q < DL ? carry[q < DL ? q : 0] : y[q - DL];
                else pa[q] = y[q];
                pb[q] = y[16 - DL + q];
            }
            const long long P = x.piece0 + 8 * c + 2 * grp;
            store_piece16<T>(base, P, pa, x.ev_lo, x.ev_hi);
            store_piece16<T>(base, P + 1, pb, x.ev_lo, x.ev_hi);
            if constexpr (DL > 0) {
#pragma unroll
                for (int q = 0; q < DL; ++q) carry[q] = y[32 - DL + q];
            }
        }
        tc_fence_before();
        mbar_arrive(&x.tempty[b]);
    }
    if constexpr (DL > 0) {  // the open piece after the last chunk
        float pa[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) pa[q] = q < DL ? carry[q < DL ? q : 0] : 0.f;
        const long long P = x.piece0 + 8 * x.nck;
        const long long e0 = P * 16;
#pragma unroll
        for (int u = 0; u < DL; ++u)
            if (e0 + u >= x.ev_lo && e0 + u <= x.ev_hi) base[e0 + u] = Elt<T>::from_f(pa[u]);
    }
}

template <typename T>
__device__ __forceinline__ void qk_rows_dispatch(int dl, const RowsCtx &x, T *base) {
    switch (dl) {
        case 0: qk_rows_epilogue<T, 0>(x, base); break;
        case 1: qk_rows_epilogue<T, 1>(x, base); break;
        case 2: qk_rows_epilogue<T, 2>(x, base); break;
        case 3: qk_rows_epilogue<T, 3>(x, base); break;
        case 4: qk_rows_epilogue<T, 4>(x, base); break;
        case 5: qk_rows_epilogue<T, 5>(x, base); break;
        case 6: qk_rows_epilogue<T, 6>(x, base); break;
        case 7: qk_rows_epilogue<T, 7>(x, base); break;
        case 8: qk_rows_epilogue<T, 8>(x, base); break;
        case 9: qk_rows_epilogue<T, 9>(x, base); break;
        case 10: qk_rows_epilogue<T, 10>(x, base); break;
        case 11: qk_rows_epilogue<T, 11>(x, base); break;
        case 12: qk_rows_epilogue<T, 12>(x, base); break;
        case 13: qk_rows_epilogue<T, 13>(x, base); break;
        case 14: qk_rows_epilogue<T, 14>(x, base); break;
        default: qk_rows_epilogue<T, 15>(x, base); break;
    }
}

template <typename T, bool kRows>
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
    const int nsplit = p.nsplit > 0 ? p.nsplit : 1;
    const int split = blockIdx.x % nsplit;
    const int a0 = (blockIdx.x / nsplit) * kBN;
    if (a0 >= nr) return;  // whole CTA leaves before any barrier or allocation
    const int kb_tile = max(a0 - g.w, 0);   // the tile's first key
    const int kb_hi = min(a0 + kBN - 1 + g.wu, nr - 1);
    const int nck_tile = (kb_hi - kb_tile + kBM) / kBM;
    constexpr int kCpc = chunks_per_cta<kRows>();
    const int c_first = split * kCpc;
    if (c_first >= nck_tile) return;
    // this CTA's chunks: [c_first, c_first + nck) of the tile
    const int kb_lo = kb_tile + c_first * kBM;
    const int nck = min(kCpc, nck_tile - c_first);

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
                        if constexpr (kRows) mma_f16_ss(d, qd, kd, idesc, k > 0);
                        else mma_f16_ss(d, kd, qd, idesc, k > 0);
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
        if constexpr (kRows) {
            const int q = quarter * 32 + lane;  // query row of this thread
            const int qq = a0 + q;
            // element coordinates relative to a 32-byte aligned base
            const uintptr_t sa = reinterpret_cast<uintptr_t>(p.S);
            T *base = reinterpret_cast<T *>(sa & ~static_cast<uintptr_t>(31));
            const long long eoff = (long long)((sa & 31) / sizeof(T));
            const long long erow = ((long long)bh * g.n + r + (long long)g.s * qq) * g.D + eoff;
            const long long e0 = erow + (kb_lo - qq + g.w);  // value 0 of chunk 0
            RowsCtx x;
            x.tfull = tfull;
            x.tempty = tempty;
            x.abort_flag = abort_flag;
            x.err = p.err;
            x.lane_base = tmem_addr(tmem, quarter * 32, 0);
            x.nck = nck;
            x.alpha = p.alpha;
            const int dl = (int)(e0 & 15);  // the same for every row of the CTA
            x.piece0 = (e0 - dl) / 16;
            if (qq < nr) {
                // the row's valid slots among this CTA's chunks (the pieces at
                // the ends of the range are shared with the neighbouring CTAs)
                x.ev_lo = max(erow + max(0, g.w - qq), e0);
                x.ev_hi = min(erow + min(g.D - 1, g.w + nr - 1 - qq), e0 + (long long)kBM * nck - 1);
            } else {
                x.ev_lo = 1;
                x.ev_hi = 0;
            }
            qk_rows_dispatch<T>(__shfl_sync(0xffffffffu, dl, 0), x, base);
        } else {
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
                uint32_t v[32];
                tmem_ld32(tmem_addr(tmem, quarter * 32, b * kBN + grp * 32), v);
                tmem_ld_wait();
                T *dst = col + (long long)(grp * 32) * stepq;
#pragma unroll
                for (int j = 0; j < 32; ++j, dst += stepq) {
                    const int q = grp * 32 + j;
                    if (q >= qlo && q <= qhi) *dst = Elt<T>::from_f(alpha * __uint_as_float(v[j]));
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[b]);
        }
        }
        // padding: slots whose key lies outside [0, nr) (the tile's first CTA)
        const T pad = Elt<T>::from_f(g.padding);
        for (int q = warp - 2; split == 0 && q < kBN; q += 4) {
            const int qq = a0 + q;
            if (qq >= nr) break;
            const int t_lo = max(0, g.w - qq);
            const int t_hi = min(g.D - 1, g.w + nr - 1 - qq);
            T *row = S + ((long long)bh * g.n + r + (long long)g.s * qq) * g.D;
            for (int t = lane; t < t_lo; t += 32) row[t] = pad;
            for (int t = t_hi + 1 + lane; t < g.D; t += 32) row[t] = pad;
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
    for (int c = threadIdx.x; c < g.hd; c += blockDim.x) arow[c] = A[c];
    __syncthreads();
    float *S = reinterpret_cast<float *>(p.out) + R * g.D;
    for (int t = threadIdx.x; t < g.D; t += blockDim.x) {
        const long long j = (long long)i + (long long)(t - g.w) * g.s;
        if (j < 0 || j >= g.n) {
            S[t] = g.padding;
        } else {
            const float *b = B + j * g.hd;
            float acc = 0.f;
            for (int c = 0; c < g.hd; ++c) acc = fmaf(arow[c], b[c], acc);
            S[t] = p.alpha * acc;
        }
    }
}

template <typename T, bool kRows>
cudaError_t launch_qk(const TmapSet &mapA, const TmapSet &mapB, const QKArgs &a0, cudaStream_t st) {
    const int tiles = (a0.g.nsub + kBN - 1) / kBN;
    // key chunks of a tile at most: its band spans kBN - 1 + w + w_upper keys
    const long long max_nck = ((long long)kBN - 1 + a0.g.w + a0.g.wu + kBM) / kBM + 1;
    QKArgs a = a0;
    constexpr int kCpc = chunks_per_cta<kRows>();
    a.nsplit = (int)((max_nck + kCpc - 1) / kCpc);
    if ((long long)tiles * a.nsplit > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)(tiles * a.nsplit), a.g.s, a.g.BH);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_band_qk_tc<T, kRows>), kSmemBytes);
    if (e != cudaSuccess) return e;
    k_band_qk_tc<T, kRows><<<grid, kThreads, kSmemBytes, st>>>(mapA, mapB, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band_qk_tc(DType dt, const TmapSet &mapA, const TmapSet &mapB,
                              const QKArgs &a, cudaStream_t st) {
    // the row-streaming epilogue needs every row of a CTA at the same offset
    // modulo 16 elements: (s*D - 1) % 16 == 0
    const bool rows = ((long long)a.g.s * a.g.D - 1) % 16 == 0;
    if (dt == kF16)
        return rows ? launch_qk<__half, true>(mapA, mapB, a, st)
                    : launch_qk<__half, false>(mapA, mapB, a, st);
    return rows ? launch_qk<__nv_bfloat16, true>(mapA, mapB, a, st)
                : launch_qk<__nv_bfloat16, false>(mapA, mapB, a, st);
}

cudaError_t launch_band_qk_f32(const DenseArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    k_band_qk_f32<<<(unsigned)rows, 128, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace swab
