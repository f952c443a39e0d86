// k_global.cu -- global tokens ("[WIP] Improve LongformerAttention
// performance", ONNX Runtime issue, item (1): one global index shared by every
// sequence of the batch).
//
// G sorted positions.  A query row i not in G attends to its band keys that
// are not in G plus all of G; a global query attends to every key.  The dense
// pieces live in companion tensors:
//   cols [BH, n, G]: every row's value at the G global keys,
//   rows [BH, G, n]: the dense rows of the G global queries.
// Every product here has G (a handful of tokens) as one of its dimensions and
// costs G*n*64 multiply-adds per slice, a few percent of the banded products;
// they run on FFMA with operands staged in shared memory.
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 7;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;       // rows per tile
constexpr int kPad = 65;        // smem row stride (floats): conflict-free column access
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> __device__ __forceinline__ float ld(const T *p) { return Elt<T>::to_f(*p); }

// rows [row0, row0 + 64) of a [n, 64] slice into smem as fp32 (zero past n)
template <typename T>
__device__ __forceinline__ void load_tile(const Geom &g, float *dst, const T *slice, int row0, int n) {
    for (int e = threadIdx.x; e < kTile * 64; e += blockDim.x) {
        const int rr = e >> 6, c = e & 63;
        const int row = row0 + rr;
        dst[rr * kPad + c] = row < n ? ld(GP(g.bnd, slice + (long long)row * 64 + c)) : 0.f;
    }
}

// the G global rows of a [n, 64] slice into smem as fp32
template <typename T>
__device__ __forceinline__ void load_global_rows(const Geom &g, float *dst, const T *slice, const GlobArgs &gl) {
    for (int e = threadIdx.x; e < gl.G * 64; e += blockDim.x) {
        const int gg = e >> 6, c = e & 63;
        dst[gg * kPad + c] = ld(GP(g.bnd, slice + (long long)gl.idx[gg] * 64 + c));
    }
}

// ---------------------------------------------------------------------------
// Dense score pieces of band_qk:
//   cols[i, g] = alpha * A[i] . B[G[g]],   rows[g, j] = alpha * A[G[g]] . B[j]
// One CTA per (64-row tile, slice).  head_dim 64 for every dtype here.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) k_glob_scores(const GlobScoreArgs p) {
    extern __shared__ float sm[];
    const GlobArgs &gl = p.gl;
    const int n = p.g.n, G = gl.G;
    const int bh = blockIdx.y, i0 = blockIdx.x * kTile;
    float *a_t = sm;                        // A tile
    float *b_t = a_t + kTile * kPad;        // B tile
    float *a_g = b_t + kTile * kPad;        // A[G]
    float *b_g = a_g + G * kPad;            // B[G]
    const T *A = reinterpret_cast<const T *>(p.A) + (long long)bh * n * 64;
    const T *B = reinterpret_cast<const T *>(p.B) + (long long)bh * n * 64;
    load_tile(p.g, a_t, A, i0, n);
    load_tile(p.g, b_t, B, i0, n);
    load_global_rows(p.g, a_g, A, gl);
    load_global_rows(p.g, b_g, B, gl);
    __syncthreads();
    T *cols = reinterpret_cast<T *>(p.cols) + (long long)bh * n * G;
    T *rows = reinterpret_cast<T *>(p.rows) + (long long)bh * G * n;
    for (int o = threadIdx.x; o < kTile * G; o += blockDim.x) {
        const int g = o % G, ii = o / G;
        if (i0 + ii >= n) continue;
        const float *x = a_t + ii * kPad, *y = b_g + g * kPad;
        float acc = 0.f;
#pragma unroll 16
        for (int c = 0; c < 64; ++c) acc = fmaf(x[c], y[c], acc);
        *GP(p.g.bnd, cols + (long long)(i0 + ii) * G + g) = Elt<T>::from_f(p.alpha * acc);
    }
    for (int o = threadIdx.x; o < kTile * G; o += blockDim.x) {
        const int jj = o % kTile, g = o / kTile;
        if (i0 + jj >= n) continue;
        const float *x = a_g + g * kPad, *y = b_t + jj * kPad;
        float acc = 0.f;
#pragma unroll 16
        for (int c = 0; c < 64; ++c) acc = fmaf(x[c], y[c], acc);
        *GP(p.g.bnd, rows + (long long)g * n + i0 + jj) = Elt<T>::from_f(p.alpha * acc);
    }
}

// ---------------------------------------------------------------------------
// Bitmap of the global positions in shared memory (n bits).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void build_bitmap(uint32_t *bm, const GlobArgs &gl, int n) {
    const int words = (n + 31) >> 5;
    for (int k = threadIdx.x; k < words; k += blockDim.x) bm[k] = 0u;
    __syncthreads();
    for (int k = threadIdx.x; k < gl.G; k += blockDim.x)
        atomicOr(&bm[gl.idx[k] >> 5], 1u << (gl.idx[k] & 31));
    __syncthreads();
}

__device__ __forceinline__ bool in_bitmap(const uint32_t *bm, long long j) {
    return (bm[j >> 5] >> (j & 31)) & 1u;
}

__device__ __forceinline__ int global_rank(const GlobArgs &gl, int j) {
    int lo = 0, hi = gl.G - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (gl.idx[mid] < j) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// Band softmax with global tokens: one warp per band row.
//   local row: max / sum over the used band slots (valid, key not global) and
//              the row's G cols values; P = 0 on unused slots; Pg cols written.
//   global row: band row and cols row written as zeros (its softmax is the
//              dense row, done by k_glob_rows_softmax).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) k_softmax_glob(const SoftmaxGlobArgs p) {
    extern __shared__ uint32_t bm[];
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    build_bitmap(bm, gl, g.n);
    const int lane = threadIdx.x & 31;
    const int rows_total = g.BH * g.n;
    const int G = gl.G;
    for (int R = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); R < rows_total;
         R += gridDim.x * (kThreads / 32)) {
        const int i = R % g.n;
        const T *srow = reinterpret_cast<const T *>(p.S) + (long long)R * g.D;
        T *prow = reinterpret_cast<T *>(p.P) + (long long)R * g.D;
        const T *sc = reinterpret_cast<const T *>(p.Scols) + (long long)R * G;
        T *pc = reinterpret_cast<T *>(p.Pcols) + (long long)R * G;
        if (in_bitmap(bm, i)) {
            for (int t = lane; t < g.D; t += 32) *GP(p.g.bnd, prow + t) = Elt<T>::from_f(0.f);
            for (int q = lane; q < G; q += 32) *GP(p.g.bnd, pc + q) = Elt<T>::from_f(0.f);
            continue;
        }
        auto used = [&](int t) {
            const long long j = (long long)i + (long long)(t - g.w) * g.s;
            return j >= 0 && j < g.n && !in_bitmap(bm, j);
        };
        // scores plus the key bias: slot t (a used slot: its key is in range)
        // and global column q (key G[q])
        const float *brow = g.kbias ? g.kbias + (size_t)(R / g.n / g.h) * g.n : nullptr;
        auto xb = [&](int t) {
            return ld(GP(p.g.bnd, srow + t)) + (brow ? __ldg(GP(p.g.bnd, brow + i + (t - g.w) * g.s)) : 0.f);
        };
        auto xc = [&](int q) { return ld(GP(p.g.bnd, sc + q)) + (brow ? __ldg(GP(p.g.bnd, brow + gl.idx[q])) : 0.f); };
        float m = -INFINITY;
        for (int t = lane; t < g.D; t += 32)
            if (used(t)) m = fmaxf(m, xb(t));
        for (int q = lane; q < G; q += 32) m = fmaxf(m, xc(q));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float mb = m * kLog2e;
        float z = 0.f;
        for (int t = lane; t < g.D; t += 32)
            if (used(t)) z += ex2(fmaf(xb(t), kLog2e, -mb));
        for (int q = lane; q < G; q += 32) z += ex2(fmaf(xc(q), kLog2e, -mb));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        const float inv = 1.f / z;
        for (int t = lane; t < g.D; t += 32)
            *GP(p.g.bnd, prow + t) = Elt<T>::from_f(used(t) ? ex2(fmaf(xb(t), kLog2e, -mb)) * inv : 0.f);
        for (int q = lane; q < G; q += 32)
            *GP(p.g.bnd, pc + q) = Elt<T>::from_f(ex2(fmaf(xc(q), kLog2e, -mb)) * inv);
        if (p.lse && lane == 0) *GP(p.g.bnd, p.lse + R) = m + logf(z);
    }
}

// Dense softmax of the G global query rows: one warp per (slice, g).
template <typename T>
__global__ void __launch_bounds__(kThreads) k_glob_rows_softmax(const SoftmaxGlobArgs p) {
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int lane = threadIdx.x & 31;
    const int W = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (W >= g.BH * gl.G) return;
    const int bh = W / gl.G, gg = W % gl.G;
    const T *x = reinterpret_cast<const T *>(p.Srows) + (long long)W * g.n;
    T *y = reinterpret_cast<T *>(p.Prows) + (long long)W * g.n;
    // the dense row's scores plus the key bias of every key
    const float *brow = g.kbias ? g.kbias + (size_t)(bh / g.h) * g.n : nullptr;
    auto xr = [&](int j) { return ld(GP(p.g.bnd, x + j)) + (brow ? __ldg(GP(p.g.bnd, brow + j)) : 0.f); };
    float m = -INFINITY;
    for (int j = lane; j < g.n; j += 32) m = fmaxf(m, xr(j));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float mb = m * kLog2e;
    float z = 0.f;
    for (int j = lane; j < g.n; j += 32) z += ex2(fmaf(xr(j), kLog2e, -mb));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float inv = 1.f / z;
    for (int j = lane; j < g.n; j += 32) *GP(p.g.bnd, y + j) = Elt<T>::from_f(ex2(fmaf(xr(j), kLog2e, -mb)) * inv);
    if (p.lse && lane == 0) *GP(p.g.bnd, p.lse + (long long)bh * g.n + gl.idx[gg]) = m + logf(z);
}

// ---------------------------------------------------------------------------
// Softmax backward with global tokens (same row structure as the forward).
//   local row: delta = sum_used P dP + sum_g Pc dPc;  dS = P (dP - delta) on
//              used slots, 0 elsewhere;  dSc = Pc (dPc - delta).
//   global row: band and cols rows written as zeros.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) k_softmax_bwd_glob(const SoftmaxGlobArgs p) {
    extern __shared__ uint32_t bm[];
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    build_bitmap(bm, gl, g.n);
    const int lane = threadIdx.x & 31;
    const int rows_total = g.BH * g.n;
    const int G = gl.G;
    for (int R = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); R < rows_total;
         R += gridDim.x * (kThreads / 32)) {
        const int i = R % g.n;
        const T *P = reinterpret_cast<const T *>(p.S) + (long long)R * g.D;
        const T *dP = reinterpret_cast<const T *>(p.S2) + (long long)R * g.D;
        T *dS = reinterpret_cast<T *>(p.P) + (long long)R * g.D;
        const T *Pc = reinterpret_cast<const T *>(p.Scols) + (long long)R * G;
        const T *dPc = reinterpret_cast<const T *>(p.S2cols) + (long long)R * G;
        T *dSc = reinterpret_cast<T *>(p.Pcols) + (long long)R * G;
        if (in_bitmap(bm, i)) {
            for (int t = lane; t < g.D; t += 32) *GP(p.g.bnd, dS + t) = Elt<T>::from_f(0.f);
            for (int q = lane; q < G; q += 32) *GP(p.g.bnd, dSc + q) = Elt<T>::from_f(0.f);
            continue;
        }
        auto used = [&](int t) {
            const long long j = (long long)i + (long long)(t - g.w) * g.s;
            return j >= 0 && j < g.n && !in_bitmap(bm, j);
        };
        float delta = 0.f;
        for (int t = lane; t < g.D; t += 32)
            if (used(t)) delta = fmaf(ld(GP(p.g.bnd, P + t)), ld(GP(p.g.bnd, dP + t)), delta);
        for (int q = lane; q < G; q += 32) delta = fmaf(ld(GP(p.g.bnd, Pc + q)), ld(GP(p.g.bnd, dPc + q)), delta);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
        for (int t = lane; t < g.D; t += 32)
            *GP(p.g.bnd, dS + t) = Elt<T>::from_f(used(t) ? ld(GP(p.g.bnd, P + t)) * (ld(GP(p.g.bnd, dP + t)) - delta) : 0.f);
        for (int q = lane; q < G; q += 32) *GP(p.g.bnd, dSc + q) = Elt<T>::from_f(ld(GP(p.g.bnd, Pc + q)) * (ld(GP(p.g.bnd, dPc + q)) - delta));
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_glob_rows_softmax_bwd(const SoftmaxGlobArgs p) {
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int lane = threadIdx.x & 31;
    const int W = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (W >= g.BH * gl.G) return;
    const T *P = reinterpret_cast<const T *>(p.Srows) + (long long)W * g.n;
    const T *dP = reinterpret_cast<const T *>(p.S2rows) + (long long)W * g.n;
    T *dS = reinterpret_cast<T *>(p.Prows) + (long long)W * g.n;
    float delta = 0.f;
    for (int j = lane; j < g.n; j += 32) delta = fmaf(ld(GP(p.g.bnd, P + j)), ld(GP(p.g.bnd, dP + j)), delta);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
    for (int j = lane; j < g.n; j += 32) *GP(p.g.bnd, dS + j) = Elt<T>::from_f(ld(GP(p.g.bnd, P + j)) * (ld(GP(p.g.bnd, dP + j)) - delta));
}

// ---------------------------------------------------------------------------
// Reductions over the sequence for the G global positions, one CTA per slice:
//   mode rows (overwrite):  out[G[g]] = alpha * sum_j W[g, j] * Y[j]
//                           (W = a rows tensor [G, n]; O and dQ of global queries)
//   mode cols (accumulate): out[G[g]] += alpha * sum_{i not in G} W[i, g] * Y[i]
//                           (W = a cols tensor [n, G]; dK and dV of global keys)
// Thread (c = channel, g = gslot + 4k) accumulates G/4 outputs in registers.
// ---------------------------------------------------------------------------
template <typename T, bool kCols>
__global__ void __launch_bounds__(kThreads) k_glob_reduce(const GlobReduceArgs p) {
    extern __shared__ float sm[];
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int n = g.n, G = gl.G;
    const int bh = blockIdx.x;
    float *y_t = sm;                  // [64][kPad]
    float *w_t = y_t + kTile * kPad;  // [64 (g)][kPad] weights for the tile: w_t[g][jj]
    uint32_t *bm = reinterpret_cast<uint32_t *>(w_t + kTile * kPad);
    if (kCols) build_bitmap(bm, gl, n);
    const T *Y = reinterpret_cast<const T *>(p.Y) + (long long)bh * n * 64;
    const T *Wt = reinterpret_cast<const T *>(p.W);
    const int c = threadIdx.x & 63, gs = threadIdx.x >> 6;  // gs in [0, 4)
    for (int gb = 0; gb < G; gb += 64) {  // blocks of 64 global positions
        const int gn = min(64, G - gb);
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;
        for (int j0 = 0; j0 < n; j0 += kTile) {
            __syncthreads();
            load_tile(p.g, y_t, Y, j0, n);
            for (int e = threadIdx.x; e < gn * kTile; e += blockDim.x) {
                const int gg = e / kTile, jj = e % kTile;
                const int j = j0 + jj;
                float wv = 0.f;
                if (j < n) {
                    if (kCols) {
                        if (!in_bitmap(bm, j)) wv = ld(GP(p.g.bnd, Wt + ((long long)bh * n + j) * G + gb + gg));
                    } else {
                        wv = ld(GP(p.g.bnd, Wt + ((long long)bh * G + gb + gg) * n + j));
                    }
                }
                w_t[gg * kPad + jj] = wv;
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int gg = gs + 4 * k;
                if (gg < gn) {
                    const float *wr = w_t + gg * kPad;
                    float a = acc[k];
#pragma unroll 8
                    for (int jj = 0; jj < kTile; ++jj) a = fmaf(wr[jj], y_t[jj * kPad + c], a);
                    acc[k] = a;
                }
            }
        }
        T *out = reinterpret_cast<T *>(p.out) + (long long)bh * n * 64;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int gg = gs + 4 * k;
            if (gg < gn) {
                T *dst = out + (long long)gl.idx[gb + gg] * 64 + c;
                const float v = p.alpha * acc[k];
                *GP(p.g.bnd, dst) = Elt<T>::from_f(kCols ? ld(GP(p.g.bnd, dst)) + v : v);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// exact fp32 band x dense products with global tokens (thread = (row, channel))
//   pv: local row i: sum over used slots + sum_g cols[i,g] V[G[g]]
//   t : key j:      sum over used (i,t) with i local + sum_g rows[g,j] Y[G[g]]
// Global query rows (pv) and global key columns (t) are finished by
// k_glob_reduce.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_band_pv_f32_glob(const DenseGlobArgs p) {
    extern __shared__ uint32_t bm[];
    const Geom &g = p.g;
    build_bitmap(bm, p.gl, g.n);
    const long long R = blockIdx.x;
    const int i = (int)(R % g.n);
    const long long bh = R / g.n;
    const int c = threadIdx.x;
    if (c >= g.hd) return;
    const float *P = reinterpret_cast<const float *>(p.A) + R * g.D;
    const float *V = reinterpret_cast<const float *>(p.B) + bh * g.n * g.hd;
    float acc = 0.f;
    if (!in_bitmap(bm, i)) {
        for (int t = 0; t < g.D; ++t) {
            const long long j = (long long)i + (long long)(t - g.w) * g.s;
            if (j < 0 || j >= g.n || in_bitmap(bm, j)) continue;
            acc = fmaf(*GP(g.bnd, P + t), *GP(g.bnd, V + j * g.hd + c), acc);
        }
        const float *cols = reinterpret_cast<const float *>(p.cols) + R * p.gl.G;
        for (int q = 0; q < p.gl.G; ++q)
            acc = fmaf(*GP(g.bnd, cols + q), *GP(g.bnd, V + (long long)p.gl.idx[q] * g.hd + c), acc);
    }
    *GP(g.bnd, reinterpret_cast<float *>(p.out) + R * g.hd + c) = p.alpha * acc;
}

__global__ void __launch_bounds__(128) k_band_t_f32_glob(const DenseGlobArgs p) {
    extern __shared__ uint32_t bm[];
    const Geom &g = p.g;
    build_bitmap(bm, p.gl, g.n);
    const long long R = blockIdx.x;
    const int j = (int)(R % g.n);
    const long long bh = R / g.n;
    const int c = threadIdx.x;
    if (c >= g.hd) return;
    const float *Bd = reinterpret_cast<const float *>(p.A) + bh * g.n * g.D;
    const float *Y = reinterpret_cast<const float *>(p.B) + bh * g.n * g.hd;
    float acc = 0.f;
    if (!in_bitmap(bm, j)) {
        for (int t = 0; t < g.D; ++t) {
            const long long i = (long long)j - (long long)(t - g.w) * g.s;
            if (i < 0 || i >= g.n || in_bitmap(bm, i)) continue;
            acc = fmaf(*GP(g.bnd, Bd + i * g.D + t), *GP(g.bnd, Y + i * g.hd + c), acc);
        }
    }
    const float *rows = reinterpret_cast<const float *>(p.rows) + bh * p.gl.G * g.n;
    for (int q = 0; q < p.gl.G; ++q)
        acc = fmaf(*GP(g.bnd, rows + (long long)q * g.n + j), *GP(g.bnd, Y + (long long)p.gl.idx[q] * g.hd + c), acc);
    *GP(g.bnd, reinterpret_cast<float *>(p.out) + R * g.hd + c) = p.alpha * acc;
}

unsigned grid_rows(long long rows_total) {
    const long long warps = rows_total;
    const long long blocks = (warps + (kThreads / 32) - 1) / (kThreads / 32);
    return (unsigned)(blocks < 4096 ? blocks : 4096);
}

size_t bitmap_bytes(int n) { return (size_t)((n + 31) / 32) * 4; }

template <typename T>
cudaError_t launch_scores_t(const GlobScoreArgs &a, cudaStream_t st) {
    const size_t smem = (size_t)(2 * kTile + 2 * a.gl.G) * kPad * sizeof(float);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_glob_scores<T>), (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.g.n + kTile - 1) / kTile, a.g.BH);
    k_glob_scores<T><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// the dense softmax of the global rows, a warp per row
template <typename T>
cudaError_t launch_rows_softmax_t(const SoftmaxGlobArgs &a, bool bwd, cudaStream_t st) {
    const unsigned rgrid = (unsigned)(((long long)a.g.BH * a.gl.G + (kThreads / 32) - 1) / (kThreads / 32));
    if (bwd)
        k_glob_rows_softmax_bwd<T><<<rgrid, kThreads, 0, st>>>(a);
    else
        k_glob_rows_softmax<T><<<rgrid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_softmax_t(const SoftmaxGlobArgs &a, bool bwd, cudaStream_t st) {
    const size_t smem = bitmap_bytes(a.g.n);
    const unsigned grid = grid_rows((long long)a.g.BH * a.g.n);
    if (bwd) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_softmax_bwd_glob<T>), (int)smem);
        if (e != cudaSuccess) return e;
        k_softmax_bwd_glob<T><<<grid, kThreads, smem, st>>>(a);
    } else {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_softmax_glob<T>), (int)smem);
        if (e != cudaSuccess) return e;
        k_softmax_glob<T><<<grid, kThreads, smem, st>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_rows_softmax_t<T>(a, bwd, st);
}

template <typename T>
cudaError_t launch_reduce_t(const GlobReduceArgs &a, bool cols, cudaStream_t st) {
    const size_t smem = (size_t)2 * kTile * kPad * sizeof(float) + (cols ? bitmap_bytes(a.g.n) : 0);
    if (cols) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_glob_reduce<T, true>), (int)smem);
        if (e != cudaSuccess) return e;
        k_glob_reduce<T, true><<<a.g.BH, kThreads, smem, st>>>(a);
    } else {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_glob_reduce<T, false>), (int)smem);
        if (e != cudaSuccess) return e;
        k_glob_reduce<T, false><<<a.g.BH, kThreads, smem, st>>>(a);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Companions of the fused forward with global tokens.  The fused kernel
// attends each query to its band keys outside G; then
//  * k_fused_glob_cols merges, into every local row, its attention over the G
//    global keys (columns): O and lse of the two disjoint key sets combine by
//    log-sum-exp;
//  * k_fused_glob_rows computes every global query's dense attention over all
//    n keys, overwriting those rows.
// The tensor-core kernels take both for G <= 64 (columns) and when the
// (16-query chunk, slice) CTAs of the rows fill the GPU; these two are the
// general forms.
// ---------------------------------------------------------------------------
struct FusedGlobArgs {
    Geom g;
    GlobArgs gl;
    float scale;
    const void *Q, *K, *V;
    void *O;
    float *lse;
};

// Thread per local row (its query and a 64-channel accumulator in
// registers), the slice's global K, V rows staged once per block and read by
// every lane at once (shared-memory broadcasts).
constexpr int kGlobColThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kGlobColThreads) k_fused_glob_cols(const FusedGlobArgs p) {
    extern __shared__ __align__(16) float sm[];
    const GlobArgs &gl = p.gl;
    const int G = gl.G, n = p.g.n, bh = blockIdx.y;
    float *kg = sm;             // [G][64]
    float *vg = kg + G * 64;    // [G][64]
    const T *Q = reinterpret_cast<const T *>(p.Q) + (long long)bh * n * 64;
    const T *K = reinterpret_cast<const T *>(p.K) + (long long)bh * n * 64;
    const T *V = reinterpret_cast<const T *>(p.V) + (long long)bh * n * 64;
    for (int e = threadIdx.x; e < G * 64; e += kGlobColThreads) {
        const int gg = e >> 6, c = e & 63;
        kg[e] = ld(GP(p.g.bnd, K + (long long)gl.idx[gg] * 64 + c));
        vg[e] = ld(GP(p.g.bnd, V + (long long)gl.idx[gg] * 64 + c));
    }
    __syncthreads();
    const int i = blockIdx.x * kGlobColThreads + threadIdx.x;
    if (i >= n) return;
    // global rows are written by k_fused_glob_rows
    int lo = 0, hi = G;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (gl.idx[mid] < i) lo = mid + 1; else hi = mid;
    }
    if (lo < G && gl.idx[lo] == i) return;
    float q[64];
    {
        const uint4 *qr = reinterpret_cast<const uint4 *>(Q + (long long)i * 64);
#pragma unroll
        for (int k = 0; k < 64 * (int)sizeof(T) / 16; ++k) {
            const uint4 v = ldg16(GP(p.g.bnd, qr + k));
            if constexpr (sizeof(T) == 2) {
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    q[8 * k + 2 * u] = lo16<T>(w[u]);
                    q[8 * k + 2 * u + 1] = hi16<T>(w[u]);
                }
            }
        }
    }
    // online softmax over the G global keys (log2 units)
    const float xs = p.scale * kLog2e;
    float m = -INFINITY, l = 0.f, acc[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) acc[c] = 0.f;
    for (int gg = 0; gg < G; ++gg) {
        const float4 *kr = reinterpret_cast<const float4 *>(kg + gg * 64);
        float d = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
            const float4 k4 = kr[c4];
            d = fmaf(q[4 * c4 + 3], k4.w, fmaf(q[4 * c4 + 2], k4.z, fmaf(q[4 * c4 + 1], k4.y, fmaf(q[4 * c4], k4.x, d))));
        }
        // plus the global key's bias (log2 units)
        const float x = p.g.kbias ? fmaf(d, xs, *GP(p.g.bnd, p.g.kbias + (size_t)(bh / p.g.h) * n + gl.idx[gg]) * kLog2e)
                                  : d * xs;
        const float mn = fmaxf(m, x);
        const float corr = ex2(m - mn);   // 0 for the first key (m = -inf)
        const float pg = ex2(x - mn);
        l = fmaf(l, corr, pg);
        const float4 *vr = reinterpret_cast<const float4 *>(vg + gg * 64);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
            const float4 v4 = vr[c4];
            acc[4 * c4] = fmaf(acc[4 * c4], corr, pg * v4.x);
            acc[4 * c4 + 1] = fmaf(acc[4 * c4 + 1], corr, pg * v4.y);
            acc[4 * c4 + 2] = fmaf(acc[4 * c4 + 2], corr, pg * v4.z);
            acc[4 * c4 + 3] = fmaf(acc[4 * c4 + 3], corr, pg * v4.w);
        }
        m = mn;
    }
    // merge with the band part (O, lse of the keys outside G)
    const long long row = (long long)bh * n + i;
    const float lse_a = *GP(p.g.bnd, p.lse + row);
    const float lse_b = m / kLog2e + logf(l);
    const float m2 = fmaxf(lse_a, lse_b);
    const float wa = expf(lse_a - m2), wb = expf(lse_b - m2);
    const float den = wa + wb;
    const float fa = wa / den, fb = wb / (l * den);
    uint4 *o4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.O) + row * 64);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint4 a = *GP(p.g.bnd, o4 + k);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
        uint32_t r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = 8 * k + 2 * u;
            r[u] = pack2<T>(fmaf(lo16<T>(w[u]), fa, acc[c] * fb), fmaf(hi16<T>(w[u]), fa, acc[c + 1] * fb));
        }
        *GP(p.g.bnd, o4 + k) = make_uint4(r[0], r[1], r[2], r[3]);
    }
    *GP(p.g.bnd, p.lse + row) = m2 + logf(den);
}

// CTA per (global query, slice): 16 key groups of 16 threads, 4 channels each
template <typename T>
__global__ void __launch_bounds__(kThreads) k_fused_glob_rows(const FusedGlobArgs p) {
    __shared__ float qs[64];
    __shared__ float red[16][66];
    const int gg = blockIdx.x, bh = blockIdx.y, n = p.g.n;
    const int i = p.gl.idx[gg];
    const T *K = reinterpret_cast<const T *>(p.K) + (long long)bh * n * 64;
    const T *V = reinterpret_cast<const T *>(p.V) + (long long)bh * n * 64;
    if (threadIdx.x < 64) qs[threadIdx.x] = ld(GP(p.g.bnd, reinterpret_cast<const T *>(p.Q) + ((long long)bh * n + i) * 64 + threadIdx.x));
    __syncthreads();
    const int kg = threadIdx.x >> 4, cq = threadIdx.x & 15;
    const float q0 = qs[4 * cq], q1 = qs[4 * cq + 1], q2 = qs[4 * cq + 2], q3 = qs[4 * cq + 3];
    const float xs = p.scale * kLog2e;
    float m = -INFINITY, l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    // the trip count is the same for every lane (the shuffles take the whole
    // warp); a group's key past the end contributes nothing
    // four keys per step (their loads in flight together), 8 bytes per load
    for (int jb = 0; jb < n; jb += 64) {
        uint2 kw[4], vw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = jb + 16 * u + kg;
            const long long off = (long long)(j < n ? j : 0) * 64 + 4 * cq;
            kw[u] = *GP(p.g.bnd, reinterpret_cast<const uint2 *>(K + off));
            vw[u] = *GP(p.g.bnd, reinterpret_cast<const uint2 *>(V + off));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool live = jb + 16 * u + kg < n;
            float d = q0 * lo16<T>(kw[u].x) + q1 * hi16<T>(kw[u].x) + q2 * lo16<T>(kw[u].y) +
                      q3 * hi16<T>(kw[u].y);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (!live) continue;
            const int j = jb + 16 * u + kg;   // plus key j's bias (log2 units)
            const float x = p.g.kbias ? fmaf(d, xs, *GP(p.g.bnd, p.g.kbias + (size_t)(bh / p.g.h) * n + j) * kLog2e)
                                      : d * xs;
            const float mn = fmaxf(m, x);
            const float corr = m == -INFINITY ? 0.f : ex2(m - mn);
            const float pj = ex2(x - mn);
            l = l * corr + pj;
            a0 = a0 * corr + pj * lo16<T>(vw[u].x);
            a1 = a1 * corr + pj * hi16<T>(vw[u].x);
            a2 = a2 * corr + pj * lo16<T>(vw[u].y);
            a3 = a3 * corr + pj * hi16<T>(vw[u].y);
            m = mn;
        }
    }
    // merge the 16 key groups
    red[kg][2 + 4 * cq] = a0;
    red[kg][3 + 4 * cq] = a1;
    red[kg][4 + 4 * cq] = a2;
    red[kg][5 + 4 * cq] = a3;
    if (cq == 0) {
        red[kg][0] = m;
        red[kg][1] = l;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int c = threadIdx.x;
        float M = -INFINITY;
        for (int k = 0; k < 16; ++k) M = fmaxf(M, red[k][0]);
        float L = 0.f, o = 0.f;
        for (int k = 0; k < 16; ++k) {
            const float f = red[k][0] == -INFINITY ? 0.f : ex2(red[k][0] - M);
            L = fmaf(red[k][1], f, L);
            o = fmaf(red[k][2 + c], f, o);
        }
        const long long row = (long long)bh * n + i;
        *GP(p.g.bnd, reinterpret_cast<T *>(p.O) + row * 64 + c) = Elt<T>::from_f(o / L);
        if (c == 0) *GP(p.g.bnd, p.lse + row) = M / kLog2e + logf(L);
    }
}

template <typename T>
cudaError_t launch_fused_glob_t(const FusedGlobArgs &a, bool cols_done, bool rows_done, cudaStream_t st) {
    const int G = a.gl.G;
    cudaError_t e;
    if (!cols_done) {
        const size_t smem = (size_t)(2 * G * 64) * sizeof(float);
        e = ensure_smem(reinterpret_cast<const void *>(k_fused_glob_cols<T>), (int)smem);
        if (e != cudaSuccess) return e;
        const dim3 grid_c((unsigned)((a.g.n + kGlobColThreads - 1) / kGlobColThreads), (unsigned)a.g.BH);
        k_fused_glob_cols<T><<<grid_c, kGlobColThreads, smem, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (rows_done) return cudaSuccess;
    // dense global rows: a CTA per (global query, slice)
    k_fused_glob_rows<T><<<dim3((unsigned)G, (unsigned)a.g.BH), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t glob_bitmap_bytes(int n) { return bitmap_bytes(n); }

cudaError_t launch_fused_glob(DType dt, const Geom &g, const GlobArgs &gl, float scale, const void *Q,
                              const void *K, const void *V, void *O, float *lse, bool cols_done,
                              bool rows_done, cudaStream_t st) {
    FusedGlobArgs a{g, gl, scale, Q, K, V, O, lse};
    if (dt == kF16) return launch_fused_glob_t<__half>(a, cols_done, rows_done, st);
    if (dt == kBF16) return launch_fused_glob_t<__nv_bfloat16>(a, cols_done, rows_done, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_glob_scores(DType dt, const GlobScoreArgs &a, cudaStream_t st) {
    if (dt == kF32) return launch_scores_t<float>(a, st);
    if (dt == kF16) return launch_scores_t<__half>(a, st);
    return launch_scores_t<__nv_bfloat16>(a, st);
}

cudaError_t launch_softmax_glob(DType dt, const SoftmaxGlobArgs &a, bool bwd, cudaStream_t st) {
    bool rows_done = false;
    cudaError_t e = cudaSuccess;
    if (launch_softmax_glob_fast(dt, a, bwd, &rows_done, st, &e)) {
        if (e != cudaSuccess || rows_done) return e;
        if (dt == kF32) return launch_rows_softmax_t<float>(a, bwd, st);
        if (dt == kF16) return launch_rows_softmax_t<__half>(a, bwd, st);
        return launch_rows_softmax_t<__nv_bfloat16>(a, bwd, st);
    }
    if (dt == kF32) return launch_softmax_t<float>(a, bwd, st);
    if (dt == kF16) return launch_softmax_t<__half>(a, bwd, st);
    return launch_softmax_t<__nv_bfloat16>(a, bwd, st);
}

cudaError_t launch_glob_reduce(DType dt, const GlobReduceArgs &a, bool cols, cudaStream_t st) {
    if (dt == kF32) return launch_reduce_t<float>(a, cols, st);
    if (dt == kF16) return launch_reduce_t<__half>(a, cols, st);
    return launch_reduce_t<__nv_bfloat16>(a, cols, st);
}

cudaError_t launch_band_f32_glob(const DenseGlobArgs &a, bool transposed, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    const size_t smem = bitmap_bytes(a.g.n);
    if (transposed) {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_band_t_f32_glob), (int)smem);
        if (e != cudaSuccess) return e;
        k_band_t_f32_glob<<<(unsigned)rows, 128, smem, st>>>(a);
    } else {
        cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_band_pv_f32_glob), (int)smem);
        if (e != cudaSuccess) return e;
        k_band_pv_f32_glob<<<(unsigned)rows, 128, smem, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace swab
