// k_global_tc.cu -- the dense global-token products of the materialised
// calls on the tensor cores (fp16 / bf16).  Global tokens as in "[WIP] Improve
// LongformerAttention performance" (ONNX Runtime issue, item (1): one index G
// shared by every sequence of the batch); each product has G as one of its
// dimensions.
//
//   scores (band_qk):  cols[i, g] = alpha * A[i] . B[G[g]]      ([n, G])
//                      rows[g, j] = alpha * A[G[g]] . B[j]      ([G, n])
//     One CTA per (128-row tile, slice, product): the tile of A (cols) or B
//     (rows) is the M side of one tcgen05 product, the gathered G rows of the
//     other tensor the N side (N = G rounded up to 16, at most 256), K = 64;
//     thread = row in the epilogue.
//   reductions over the sequence (band_pv / band_t, global outputs):
//     rows mode:  out[G[g]]  = alpha * sum_j W[g, j] Y[j]           (W [G, n])
//     cols mode:  out[G[g]] += alpha * sum_{i not in G} W[i, g] Y[i] (W [n, G])
//     One CTA per (slice, block of 128 global positions): M = the block's
//     positions (zero past G), N = 64 channels, K = the sequence in chunks of
//     64; W chunks are staged by the threads (K-major for rows, MN-major for
//     cols, global rows of W zeroed in cols mode), Y chunks arrive by TMA,
//     two stages.  The fp32 accumulator stays in tensor memory.
// fp32 keeps the FFMA kernels of k_global.cu.
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 8;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kRows = 128;        // M of every product here
constexpr int kChunk = 64;        // sequence positions per reduction chunk (K)
constexpr int kThreads = 128;     // thread = TMEM lane / M row in the epilogues

// byte offset of 16-byte piece `c` of 128-byte line `row` in a 128-B-swizzled tile
__device__ __forceinline__ uint32_t sw128(int row, int c) { return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4)); }

__device__ __forceinline__ uint32_t tmem_cols_for(int n) {
    uint32_t c = 32;
    while (c < (uint32_t)n) c <<= 1;
    return c;
}

// ---------------------------------------------------------------------------
// score pieces
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    k_glob_scores_tc(const __grid_constant__ TmapSet mapA, const __grid_constant__ TmapSet mapB,
                     const GlobScoreArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *xt = base;                    // 128 rows x 64, TMA
    uint8_t *yg = base + kRows * 128;      // Gp gathered rows x 64, swizzled by the threads
    __shared__ uint64_t bars[2];           // 0: tile landed, 1: product done
    __shared__ uint32_t tmem_holder;
    __shared__ int abort_flag;
    const int G = p.gl.G, Gp = (G + 15) & ~15;
    const int n = p.g.n, bh = blockIdx.y, i0 = blockIdx.x * kRows;
    const bool rows = blockIdx.z == 1;      // rows^T: M = keys of B, N = A[G]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ncols = tmem_cols_for(Gp);
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_holder, ncols);
        tmem_relinquish();
    }
    // the gathered rows (of B for cols, of A for rows), zero past G
    const T *ysrc = reinterpret_cast<const T *>(rows ? p.A : p.B) + (size_t)bh * n * 64;
    for (int e = threadIdx.x; e < Gp * 8; e += kThreads) {
        const int q = e >> 3, c = e & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (q < G) v = *GP(p.g.bnd, reinterpret_cast<const uint4 *>(ysrc + (size_t)p.gl.idx[q] * 64 + 8 * c));
        *reinterpret_cast<uint4 *>(yg + sw128(q, c)) = v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    unsigned *err = p.err;
    bool ok = true;
    if (threadIdx.x == 0) {
        const CUtensorMap *m = rows ? &mapB.m[0] : &mapA.m[0];
        mbar_arrive_expect_tx(&bars[0], kRows * 128);
        tma_load_3d(xt, m, &bars[0], 0, i0, bh);
        ok = mbar_wait(&bars[0], 0, &abort_flag, err);
        if (ok) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t idesc = idesc_f16(kRows, Gp, kBf16, false, false);
            const uint64_t da = sdesc_sw128(smem_u32(xt), 16, 1024), db = sdesc_sw128(smem_u32(yg), 16, 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_f16_ss(tmem, da + 2 * k, db + 2 * k, idesc, k > 0);
            mma_commit(&bars[1]);
        }
    }
    // every thread waits for the product (or the abort)
    ok = mbar_wait(&bars[1], 0, &abort_flag, err);
    tc_fence_after();
    const int m = warp * 32 + lane, row = i0 + m;
    if (__all_sync(0xffffffffu, ok)) {
        for (int g0 = 0; g0 < Gp; g0 += 32) {
            uint32_t v[32];
            if (g0 + 32 <= (int)ncols) {
                tmem_ld32(tmem_addr(tmem, warp * 32, g0), v);
                tmem_ld_wait();
            }
            if (row < n) {
                if (!rows) {
                    T *dst = reinterpret_cast<T *>(p.cols) + ((size_t)bh * n + row) * G;
                    for (int k = 0; k < 32 && g0 + k < G; ++k)
                        *GP(p.g.bnd, dst + g0 + k) = Elt<T>::from_f(p.alpha * __uint_as_float(v[k]));
                } else {
                    T *dst = reinterpret_cast<T *>(p.rows) + (size_t)bh * G * n + row;
                    for (int k = 0; k < 32 && g0 + k < G; ++k)
                        *GP(p.g.bnd, dst + (size_t)(g0 + k) * n) = Elt<T>::from_f(p.alpha * __uint_as_float(v[k]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, ncols);
    }
}

// ---------------------------------------------------------------------------
// reductions over the sequence
// ---------------------------------------------------------------------------
constexpr int kATile = kRows * 128;        // 16 KB: W chunk (rows: 128 x 64 K-major; cols: 64 lines x 128 M)
constexpr int kBTile = kChunk * 128;       // 8 KB: Y chunk, 64 rows x 64
constexpr int kStageBytes = kATile + kBTile;

// The sequence is split over a cluster of kSplit CTAs (one slice and 128
// global positions a cluster): each CTA sums its share of the chunks into
// tensor memory, the partial sums meet in shared memory, and each CTA of the
// cluster finishes 1/kSplit of the rows from every CTA's partial (read through
// distributed shared memory).  One CTA a slice walked the whole sequence
// alone and took 0.28 ms at b*h = 144, n = 4096.
constexpr int kSplit = 8;
constexpr int kPartStride = 65;   // floats a row of the partial (bank-conflict free)

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer_f32(const float *local, int rank) {
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
    return v;
}

template <typename T, bool kCols>
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kThreads, 1)
    k_glob_reduce_tc(const __grid_constant__ TmapSet mapY, const GlobReduceArgs p, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint32_t *bm = reinterpret_cast<uint32_t *>(base + 2 * kStageBytes);   // cols: global positions
    float *part = reinterpret_cast<float *>(base);   // the partial sums, once the stages are idle
    __shared__ uint64_t full[2], empty[2], done;
    __shared__ uint32_t tmem_holder;
    __shared__ int abort_flag;
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int rank = blockIdx.x;   // rank in the cluster = share of the sequence
    const int n = g.n, G = gl.G, bh = blockIdx.y, q0 = blockIdx.z * kRows;
    const int qn = min(kRows, G - q0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (kCols) {
        for (int k = threadIdx.x; k < (n + 31) / 32; k += kThreads) bm[k] = 0u;
        __syncthreads();
        for (int k = threadIdx.x; k < G; k += kThreads) atomicOr(&bm[gl.idx[k] >> 5], 1u << (gl.idx[k] & 31));
    }
    // zero both W stages once: rows mode writes lines q < qn only, cols mode
    // every line but only columns < qn
    for (int e = threadIdx.x; e < 2 * kStageBytes / 16; e += kThreads)
        reinterpret_cast<uint4 *>(base)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) {
        tmem_alloc(&tmem_holder, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    const T *W = reinterpret_cast<const T *>(p.W);
    const int nch = (n + kChunk - 1) / kChunk;
    const int cps = (nch + kSplit - 1) / kSplit;
    const int c0 = rank * cps, c1 = min(nch, c0 + cps);
    constexpr bool kBf16 = !std::is_same<T, __half>::value;
    // A: rows mode K-major (line = global position, 64 sequence elements);
    // cols mode MN-major (line = sequence position, 64 global positions; the
    // two 64-position halves of M sit kATile / 2 apart).  B = Y rows, MN-major.
    const uint32_t idesc = idesc_f16(kRows, 64, kBf16, kCols, true);
    bool ok = true;
    for (int c = c0; c < c1 && ok; ++c) {
        const int lc = c - c0;
        const int st = lc & 1;
        uint8_t *at = base + st * kStageBytes, *btile = at + kATile;
        // the stage was last read by the products of chunk lc - 2
        if (lc >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((lc >> 1) - 1) & 1, &abort_flag, err)) &&
                          ok;
        ok = __syncthreads_and(ok);
        if (!ok) break;
        const int j0 = c * kChunk;
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&full[st], kBTile);
            tma_load_3d(btile, &mapY.m[0], &full[st], 0, j0, bh);
        }
        // 16-byte pieces of 8 consecutive W elements: one 16-byte load where
        // they are in range and aligned, else element by element
        auto piece = [&](const T *src, int cnt) -> uint4 {
            if (cnt >= 8 && (reinterpret_cast<uintptr_t>(src) & 15) == 0)
                return *GP(g.bnd, reinterpret_cast<const uint4 *>(src));
            float f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) f[u] = u < cnt ? Elt<T>::to_f(*GP(g.bnd, src + u)) : 0.f;
            return make_uint4(pack2<T>(f[0], f[1]), pack2<T>(f[2], f[3]), pack2<T>(f[4], f[5]),
                              pack2<T>(f[6], f[7]));
        };
        if constexpr (!kCols) {
            // line q: W[q0 + q, j0 .. j0 + 63]
            for (int e = threadIdx.x; e < qn * (kChunk / 8); e += kThreads) {
                const int q = e >> 3, c8 = e & 7, j = j0 + 8 * c8;
                const uint4 v = j < n ? piece(W + ((size_t)bh * G + q0 + q) * n + j, n - j)
                                      : make_uint4(0u, 0u, 0u, 0u);
                sts16(smem_u32(at + sw128(q, c8)), v);
            }
        } else {
            // line jj: W[j0 + jj, q0 .. q0 + 127], zero at a global row
            const int qp = (qn + 7) / 8;
            for (int e = threadIdx.x; e < kChunk * qp; e += kThreads) {
                const int jj = e / qp, c8 = e % qp, j = j0 + jj, q = 8 * c8;
                const bool use = j < n && !((bm[j >> 5] >> (j & 31)) & 1u);
                const uint4 v = use ? piece(W + ((size_t)bh * n + j) * G + q0 + q, qn - q)
                                    : make_uint4(0u, 0u, 0u, 0u);
                uint8_t *half = at + (q >> 6) * (kATile / 2);
                sts16(smem_u32(half + sw128(jj, (q & 63) >> 3)), v);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            ok = mbar_wait(&full[st], (lc >> 1) & 1, &abort_flag, err);
            if (ok) {
                tc_fence_after();
                const uint64_t da = kCols ? sdesc_sw128(smem_u32(at), kATile / 2, 1024) : sdesc_sw128(smem_u32(at), 16, 1024);
                const uint64_t db = sdesc_sw128(smem_u32(btile), 1024, 1024);
#pragma unroll
                for (int k = 0; k < kChunk / 16; ++k) {
                    // K step k = sequence positions 16k .. 16k + 15
                    const uint64_t ak = kCols ? da + (uint64_t)((2048 * k) >> 4) : da + 2 * k;
                    mma_f16_ss(tmem, ak, db + (uint64_t)((2048 * k) >> 4), idesc, (lc > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&empty[st]);
                if (c == c1 - 1) mma_commit(&done);
            }
        }
    }
    ok = __syncthreads_and(ok);
    const bool any = c1 > c0;
    bool fin = ok && (!any || mbar_wait(&done, 0, &abort_flag, err));
    tc_fence_after();
    // this CTA's partial sums (zero without chunks) into shared memory; the
    // stages are idle once `done` has fired
    const int q = warp * 32 + lane;
    const bool have = __all_sync(0xffffffffu, fin) && any;
    for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        if (have) {
            tmem_ld32(tmem_addr(tmem, warp * 32, 32 * h), v);
            tmem_ld_wait();
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) part[q * kPartStride + 32 * h + k] = have ? __uint_as_float(v[k]) : 0.f;
    }
    cluster_sync();
    // rows [r0, r1) of the 128: the sum over the cluster's partials
    const int per = (qn + kSplit - 1) / kSplit;
    const int r0 = min(qn, rank * per), r1 = min(qn, r0 + per);
    for (int e = threadIdx.x; e < (r1 - r0) * 64; e += kThreads) {
        const int qq = r0 + (e >> 6), ch = e & 63;
        const float *loc = part + qq * kPartStride + ch;
        float acc = 0.f;
#pragma unroll
        for (int rr = 0; rr < kSplit; ++rr) acc += ld_peer_f32(loc, rr);
        T *dst = reinterpret_cast<T *>(p.out) + ((size_t)bh * n + gl.idx[q0 + qq]) * 64 + ch;
        const float x = p.alpha * acc;
        *GP(g.bnd, dst) = Elt<T>::from_f(kCols ? Elt<T>::to_f(*GP(g.bnd, dst)) + x : x);
    }
    // no CTA leaves while another still reads its partial
    cluster_sync();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, 64);
    }
}

}  // namespace

cudaError_t launch_glob_scores_tc(DType dt, const TmapSet &mapA, const TmapSet &mapB, const GlobScoreArgs &a,
                                  cudaStream_t st) {
    if (a.gl.G < 1 || a.gl.G > 256 || a.g.BH > 65535) return cudaErrorInvalidValue;
    const int Gp = (a.gl.G + 15) & ~15;
    const size_t smem = (size_t)kRows * 128 + (size_t)Gp * 128 + 1024;
    const dim3 grid((a.g.n + kRows - 1) / kRows, a.g.BH, 2);
    if (dt == kF16) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_glob_scores_tc<__half>), (int)smem);
        if (e != cudaSuccess) return e;
        k_glob_scores_tc<__half><<<grid, kThreads, smem, st>>>(mapA, mapB, a);
    } else {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_glob_scores_tc<__nv_bfloat16>), (int)smem);
        if (e != cudaSuccess) return e;
        k_glob_scores_tc<__nv_bfloat16><<<grid, kThreads, smem, st>>>(mapA, mapB, a);
    }
    return cudaGetLastError();
}

cudaError_t launch_glob_reduce_tc(DType dt, const TmapSet &mapY, const GlobReduceArgs &a, bool cols, unsigned *err,
                                  cudaStream_t st) {
    if (a.gl.G < 1 || a.g.BH > 65535) return cudaErrorInvalidValue;
    const size_t smem = 2 * (size_t)kStageBytes + 1024 + (cols ? (size_t)((a.g.n + 31) / 32) * 4 : 0);
    const dim3 grid(kSplit, a.g.BH, (a.gl.G + kRows - 1) / kRows);
    cudaError_t e;
#define SWAB_LAUNCH_RED(TT, CC)                                                                              \
    e = ensure_smem(reinterpret_cast<const void *>(k_glob_reduce_tc<TT, CC>), (int)smem);                    \
    if (e != cudaSuccess) return e;                                                                          \
    k_glob_reduce_tc<TT, CC><<<grid, kThreads, smem, st>>>(mapY, a, err);
    if (dt == kF16) {
        if (cols) { SWAB_LAUNCH_RED(__half, true) } else { SWAB_LAUNCH_RED(__half, false) }
    } else {
        if (cols) { SWAB_LAUNCH_RED(__nv_bfloat16, true) } else { SWAB_LAUNCH_RED(__nv_bfloat16, false) }
    }
#undef SWAB_LAUNCH_RED
    return cudaGetLastError();
}

}  // namespace swab
