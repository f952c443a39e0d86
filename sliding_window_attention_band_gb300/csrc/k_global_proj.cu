// k_global_proj.cu -- global queries with their own projections (ONNX Runtime
// issue "[WIP] Improve LongformerAttention performance", item (3): the
// global_q projection computed only for the G global tokens -- a compact Qg --
// with separate global key and value projections Kg, Vg over every position).
//
//   forward:  Og[g] = softmax_j(scale Qg[g].Kg[j]) Vg,  lseg[g]
//   backward: delta_g = dOg[g].Og[g];  ds_gj = p_gj (dOg[g].Vg[j] - delta_g)
//             dQg = scale ds Kg,  dKg = scale ds^T Qg,  dVg = p^T dOg
//
// G is a handful of tokens, so every product has G as one dimension.  The
// 16-bit paths run on the tensor cores with the keys as the M dimension: one
// CTA per (128-key tile, slice) computes S^T = Kg Qg^T (N = 16 queries per
// chunk) into tensor memory; the forward writes a (max, sum, output) partial
// per tile that a second kernel merges, the backward forms dVg, dKg (one
// writer per key row) and per-tile dQg partials summed by a second kernel in
// a fixed order.  fp32 runs FFMA kernels on operands staged in shared memory
// (256-key chunks in the forward, 64-key tiles in the backward).  Partials
// live in the caller's workspace.
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 9;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kThreads = 256;
constexpr int kGC = 16;          // global queries per chunk
constexpr int kKT = 64;          // keys per tile
constexpr int kPad = 68;         // smem row stride (floats): 16-byte rows, 8 rows hit 8 bank groups
constexpr int kChunkKeys = 256;  // forward: keys per CTA
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// acc += a * v (four channels)
__device__ __forceinline__ void axpy4(float4 &acc, float a, const float4 v) {
    acc.x = fmaf(a, v.x, acc.x);
    acc.y = fmaf(a, v.y, acc.y);
    acc.z = fmaf(a, v.z, acc.z);
    acc.w = fmaf(a, v.w, acc.w);
}

// rows [row0, row0 + nrows) of a [*, 64] array into smem as fp32 rows of kPad,
// 16 bytes per load (rows at or past `limit` are zero)
template <typename T>
__device__ __forceinline__ void load_rows(const GlobalProjArgs &p, float *dst, const T *src, int row0, int nrows, int limit) {
    constexpr int V = 16 / sizeof(T);   // elements per 16-byte load
    for (int e = threadIdx.x; e < nrows * (64 / V); e += kThreads) {
        const int r = e / (64 / V), c0 = (e % (64 / V)) * V;
        const int row = row0 + r;
        float *d = dst + r * kPad + c0;
        if (row < limit) {
            const uint4 v = ldg16(GP(p.bnd, reinterpret_cast<const uint4 *>(src + (long long)row * 64 + c0)));
            if constexpr (sizeof(T) == 4) {
                *reinterpret_cast<float4 *>(d) = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                                             __uint_as_float(v.z), __uint_as_float(v.w));
            } else {
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                *reinterpret_cast<float4 *>(d) = make_float4(lo16<T>(w[0]), hi16<T>(w[0]), lo16<T>(w[1]),
                                                             hi16<T>(w[1]));
                *reinterpret_cast<float4 *>(d + 4) = make_float4(lo16<T>(w[2]), hi16<T>(w[2]),
                                                                 lo16<T>(w[3]), hi16<T>(w[3]));
            }
        } else {
#pragma unroll
            for (int k = 0; k < V; ++k) d[k] = 0.f;
        }
    }
}

// A 64 x 64 tile's 16-byte pieces held in registers between its global load
// and its shared-memory store (the next tile is fetched while the current one
// is used): thread x holds pieces x, x + 256, ...
template <typename T> struct TileRegs {
    static constexpr int kPer = 64 * 64 * (int)sizeof(T) / 16 / kThreads;
    uint4 v[kPer];
};

template <typename T>
__device__ __forceinline__ void fetch_tile(const GlobalProjArgs &p, TileRegs<T> &r, const T *src, int row0, int limit) {
    constexpr int V = 16 / sizeof(T), PR = 64 / V;   // elements per piece, pieces per row
#pragma unroll
    for (int k = 0; k < TileRegs<T>::kPer; ++k) {
        const int e = threadIdx.x + kThreads * k;
        const int row = row0 + e / PR;
        r.v[k] = row < limit ? ldg16(GP(p.bnd, reinterpret_cast<const uint4 *>(src + (long long)row * 64 + (e % PR) * V)))
                             : make_uint4(0, 0, 0, 0);
    }
}

template <typename T>
__device__ __forceinline__ void store_tile(float *dst, const TileRegs<T> &r) {
    constexpr int V = 16 / sizeof(T), PR = 64 / V;
#pragma unroll
    for (int k = 0; k < TileRegs<T>::kPer; ++k) {
        const int e = threadIdx.x + kThreads * k;
        float *d = dst + (e / PR) * kPad + (e % PR) * V;
        const uint4 v = r.v[k];
        if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float4 *>(d) = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                                         __uint_as_float(v.z), __uint_as_float(v.w));
        } else {
            *reinterpret_cast<float4 *>(d) = make_float4(lo16<T>(v.x), hi16<T>(v.x), lo16<T>(v.y), hi16<T>(v.y));
            *reinterpret_cast<float4 *>(d + 4) =
                make_float4(lo16<T>(v.z), hi16<T>(v.z), lo16<T>(v.w), hi16<T>(v.w));
        }
    }
}

// ---------------------------------------------------------------------------
// forward partials: CTA (key chunk, query chunk, slice)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) k_gproj_fwd(const GlobalProjArgs p) {
    __shared__ __align__(16) float qs[kGC * kPad], ks[kKT * kPad], vs[kKT * kPad], ps[kGC * kPad];
    const int kc = blockIdx.x, gc = blockIdx.y, bh = blockIdx.z;
    const int G = p.G, n = p.n, t = threadIdx.x;
    const int g = t >> 4, sub = t & 15;            // query g of the chunk; key / channel phase
    const T *Qg = reinterpret_cast<const T *>(p.Qg) + (long long)bh * G * 64;
    const T *Kg = reinterpret_cast<const T *>(p.Kg) + (long long)bh * n * 64;
    const T *Vg = reinterpret_cast<const T *>(p.Vg) + (long long)bh * n * 64;
    load_rows(p, qs, Qg, gc * kGC, kGC, G);
    const float xs = p.scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);   // channels 4 sub .. + 3
    const int k0 = kc * kChunkKeys, k1 = min(n, k0 + kChunkKeys);
    TileRegs<T> kr, vr;
    fetch_tile(p, kr, Kg, k0, n);
    fetch_tile(p, vr, Vg, k0, n);
    for (int j0 = k0; j0 < k1; j0 += kKT) {
        __syncthreads();   // the previous tile's readers are done
        store_tile(ks, kr);
        store_tile(vs, vr);
        if (j0 + kKT < k1) {   // the next tile's loads fly during this tile's products
            fetch_tile(p, kr, Kg, j0 + kKT, n);
            fetch_tile(p, vr, Vg, j0 + kKT, n);
        }
        __syncthreads();
        float s[4] = {0.f, 0.f, 0.f, 0.f}, tmax = -INFINITY;
#pragma unroll 4
        for (int c = 0; c < 64; c += 4) {
            const float4 q4 = lds4(qs + g * kPad + c);
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] = dot4(q4, lds4(ks + (sub + 16 * u) * kPad + c), s[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            s[u] = j0 + sub + 16 * u < n ? s[u] * xs : -INFINITY;   // log2 units
            tmax = fmaxf(tmax, s[u]);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float mn = fmaxf(m, tmax);           // finite: the tile has a key < n
        const float corr = m == -INFINITY ? 0.f : ex2(m - mn);
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float pv = ex2(s[u] - mn);
            ps[g * kPad + sub + 16 * u] = pv;
            psum += pv;
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * corr + psum;
        m = mn;
        __syncthreads();
        acc.x *= corr;
        acc.y *= corr;
        acc.z *= corr;
        acc.w *= corr;
#pragma unroll 4
        for (int j = 0; j < kKT; j += 4) {
            const float4 p4 = lds4(ps + g * kPad + j);
            const float *vr = vs + j * kPad + 4 * sub;
            axpy4(acc, p4.x, lds4(vr));
            axpy4(acc, p4.y, lds4(vr + kPad));
            axpy4(acc, p4.z, lds4(vr + 2 * kPad));
            axpy4(acc, p4.w, lds4(vr + 3 * kPad));
        }
    }
    const int gg = gc * kGC + g;
    if (gg >= G) return;
    // partial of (slice, chunk, query): [m (log2 units), l, acc[64]]
    float *part = p.ws + (((long long)bh * p.nchunks + kc) * G + gg) * 66;
    if (sub == 0) {
        *GP(p.bnd, part) = m;
        *GP(p.bnd, part + 1) = l;
    }
    *GP(p.bnd, part + 2 + 4 * sub) = acc.x;
    *GP(p.bnd, part + 3 + 4 * sub) = acc.y;
    *GP(p.bnd, part + 4 + 4 * sub) = acc.z;
    *GP(p.bnd, part + 5 + 4 * sub) = acc.w;
}

// merge the chunks: a warp per (slice, query); lane k < nchunks reads chunk
// k's (max, sum) at once, then every lane merges two channels over the chunks
// with eight loads in flight
template <typename T>
__global__ void __launch_bounds__(kThreads) k_gproj_combine(const GlobalProjArgs p) {
    const long long bg = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);   // bh*G + g
    if (bg >= (long long)p.BH * p.G) return;
    const int lane = threadIdx.x & 31;
    const long long bh = bg / p.G, gg = bg - bh * p.G;
    const float *base = p.ws + ((long long)bh * p.nchunks * p.G + gg) * 66;
    const long long step = (long long)p.G * 66;     // next chunk of the same query
    float M = -INFINITY;
    for (int k = lane; k < p.nchunks; k += 32) M = fmaxf(M, *GP(p.bnd, base + k * step));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int k = lane; k < p.nchunks; k += 32)
        L = fmaf(*GP(p.bnd, base + k * step + 1), ex2(*GP(p.bnd, base + k * step) - M), L);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    float o0 = 0.f, o1 = 0.f;
    int k = 0;
    for (; k + 8 <= p.nchunks; k += 8) {
        float f[8], a[8], b[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float *c = base + (k + u) * step;
            f[u] = *GP(p.bnd, c);
            a[u] = *GP(p.bnd, c + 2 + 2 * lane);
            b[u] = *GP(p.bnd, c + 3 + 2 * lane);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float w = ex2(f[u] - M);
            o0 = fmaf(a[u], w, o0);
            o1 = fmaf(b[u], w, o1);
        }
    }
    for (; k < p.nchunks; ++k) {
        const float *c = base + k * step;
        const float w = ex2(*GP(p.bnd, c) - M);
        o0 = fmaf(*GP(p.bnd, c + 2 + 2 * lane), w, o0);
        o1 = fmaf(*GP(p.bnd, c + 3 + 2 * lane), w, o1);
    }
    const float inv = 1.f / L;
    T *o = reinterpret_cast<T *>(p.Og) + bg * 64 + 2 * lane;
    *GP(p.bnd, o) = Elt<T>::from_f(o0 * inv);
    *GP(p.bnd, o + 1) = Elt<T>::from_f(o1 * inv);
    if (lane == 0 && p.lseg) *GP(p.bnd, p.lseg + bg) = M / kLog2e + logf(L);
}

// ---------------------------------------------------------------------------
// backward, fp32 operands (FFMA): CTA (64-key tile, slice) over every global query
// ---------------------------------------------------------------------------
// shared memory of the backward (floats): K, V tiles; Qg, dOg chunks; p, ds
// of the chunk; lse, delta of the chunk
constexpr int kBwdSmemFloats = 2 * kKT * kPad + 4 * kGC * kPad + 2 * kGC;

template <typename T>
__global__ void __launch_bounds__(kThreads) k_gproj_bwd(const GlobalProjArgs p) {
    extern __shared__ __align__(16) float smb[];
    float *ks = smb, *vs = ks + kKT * kPad, *qs = vs + kKT * kPad, *dos = qs + kGC * kPad;
    float *ps = dos + kGC * kPad, *dss = ps + kGC * kPad, *lse_s = dss + kGC * kPad,
          *del_s = lse_s + kGC;
    const int kt = blockIdx.x, bh = blockIdx.y;
    const int G = p.G, n = p.n, t = threadIdx.x;
    const int g = t >> 4, sub = t & 15;
    const int j0 = kt * kKT;
    const T *Qg = reinterpret_cast<const T *>(p.Qg) + (long long)bh * G * 64;
    const T *Og = reinterpret_cast<const T *>(p.Og) + (long long)bh * G * 64;
    const T *dOg = reinterpret_cast<const T *>(p.dOg) + (long long)bh * G * 64;
    const T *Kg = reinterpret_cast<const T *>(p.Kg) + (long long)bh * n * 64;
    const T *Vg = reinterpret_cast<const T *>(p.Vg) + (long long)bh * n * 64;
    load_rows(p, ks, Kg, j0, kKT, n);
    load_rows(p, vs, Vg, j0, kKT, n);
    // dK, dV of key jr = t / 4, channels 16 (t % 4) .. + 16
    const int jr = t >> 2, cq = (t & 3) * 16;
    float dk[16], dv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) dk[k] = dv[k] = 0.f;
    const float xs = p.scale * kLog2e;
    for (int g0 = 0; g0 < G; g0 += kGC) {
        __syncthreads();   // the previous chunk's readers are done
        load_rows(p, qs, Qg, g0, kGC, G);
        load_rows(p, dos, dOg, g0, kGC, G);
        if (t < kGC) lse_s[t] = g0 + t < G ? *GP(p.bnd, p.lseg + (long long)bh * G + g0 + t) * kLog2e : 0.f;
        // delta_g = dOg[g].Og[g]: 16 threads per query, 4 channels each
        {
            float d = 0.f;
            if (g0 + g < G) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = sub + 16 * u;
                    d = fmaf(Elt<T>::to_f(*GP(p.bnd, dOg + (long long)(g0 + g) * 64 + c)),
                             Elt<T>::to_f(*GP(p.bnd, Og + (long long)(g0 + g) * 64 + c)), d);
                }
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (sub == 0) del_s[g] = d;
        }
        __syncthreads();
        // p and ds of (query g, keys sub + 16 u)
        {
            float sd[4] = {0.f, 0.f, 0.f, 0.f}, pd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int c = 0; c < 64; c += 4) {
                const float4 q4 = lds4(qs + g * kPad + c), o4 = lds4(dos + g * kPad + c);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = sub + 16 * u;
                    sd[u] = dot4(q4, lds4(ks + j * kPad + c), sd[u]);
                    pd[u] = dot4(o4, lds4(vs + j * kPad + c), pd[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = sub + 16 * u;
                const bool live = g0 + g < G && j0 + j < n;
                const float pr = live ? ex2(sd[u] * xs - lse_s[g]) : 0.f;
                ps[g * kPad + j] = pr;
                dss[g * kPad + j] = pr * (pd[u] - del_s[g]);
            }
        }
        __syncthreads();
        // dQg partial of (query g, channels 4 sub .. + 3) over this tile's keys
        if (g0 + g < G) {
            float4 dq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int j = 0; j < kKT; j += 4) {
                const float4 d4 = lds4(dss + g * kPad + j);
                const float *kr = ks + j * kPad + 4 * sub;
                axpy4(dq, d4.x, lds4(kr));
                axpy4(dq, d4.y, lds4(kr + kPad));
                axpy4(dq, d4.z, lds4(kr + 2 * kPad));
                axpy4(dq, d4.w, lds4(kr + 3 * kPad));
            }
            float *part = p.ws + (((long long)bh * p.nchunks + kt) * G + g0 + g) * 64 + 4 * sub;
            *GP(p.bnd, reinterpret_cast<float4 *>(part)) =
                make_float4(p.scale * dq.x, p.scale * dq.y, p.scale * dq.z, p.scale * dq.w);
        }
        // dK[jr] += scale sum_g ds_g,jr Qg[g];  dV[jr] += sum_g p_g,jr dOg[g]
#pragma unroll 2
        for (int q = 0; q < kGC; ++q) {
            const float dsv = dss[q * kPad + jr], pv = ps[q * kPad + jr];
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                const float4 q4 = lds4(qs + q * kPad + cq + k), o4 = lds4(dos + q * kPad + cq + k);
                dk[k] = fmaf(dsv, q4.x, dk[k]);
                dk[k + 1] = fmaf(dsv, q4.y, dk[k + 1]);
                dk[k + 2] = fmaf(dsv, q4.z, dk[k + 2]);
                dk[k + 3] = fmaf(dsv, q4.w, dk[k + 3]);
                dv[k] = fmaf(pv, o4.x, dv[k]);
                dv[k + 1] = fmaf(pv, o4.y, dv[k + 1]);
                dv[k + 2] = fmaf(pv, o4.z, dv[k + 2]);
                dv[k + 3] = fmaf(pv, o4.w, dv[k + 3]);
            }
        }
    }
    if (j0 + jr >= n) return;
    T *dK = reinterpret_cast<T *>(p.dKg) + ((long long)bh * n + j0 + jr) * 64 + cq;
    T *dV = reinterpret_cast<T *>(p.dVg) + ((long long)bh * n + j0 + jr) * 64 + cq;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        *GP(p.bnd, dK + k) = Elt<T>::from_f(p.scale * dk[k]);
        *GP(p.bnd, dV + k) = Elt<T>::from_f(dv[k]);
    }
}

// ---------------------------------------------------------------------------
// backward on the tensor cores: CTA (128-key tile, slice), every global query
// in chunks of 16.  With the keys as the M dimension every product has a
// tcgen05 shape (M = 128):
//   S^T  = Kg Qg_c^T,  dP^T = Vg dOg_c^T          (N = 16, K = 64)
//   dVg += P_c^T dOg_c, dKg += dS_c^T Qg_c         (N = 64, K = 16)
//   dQg_c^T = Kg^T dS_c                           (K = 128 keys; Kg read as an
//        MN-major A of 128 rows whose second 64-row block is the V tile: those
//        32 output lanes are never read)
// Warp 0 loads (TMA), warp 1 owns tensor memory and issues the products,
// warps 2-5 (lane = key) turn S^T, dP^T into P and dS and read the results.
// ---------------------------------------------------------------------------
constexpr int kTcThreads = 192;
constexpr int kTcKeys = 128;
constexpr uint32_t kTcTmemCols = 256;
constexpr uint32_t kColS = 0, kColDP = 16, kColDQ = 32, kColDV = 64, kColDK = 128;
constexpr int kTile16 = kTcKeys * 128;   // a 128 x 64 16-bit tile, bytes

// shared memory of the tensor-core backward for nch query chunks (bytes)
__host__ __device__ constexpr int tc_bwd_smem(int nch) {
    return 1024 /* alignment */ + 2 * kTile16 /* K, V */ + 2 * nch * 2048 /* Qg, dOg */ +
           2 * kTile16 /* P, dS (keys x queries) */ + 2 * 2048 /* dS (queries x keys) */ +
           2 * 256 * 4 /* lse, delta */ + 256 /* barriers, flags */;
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_gproj_bwd_tc(const __grid_constant__ TmapSet mapK, const __grid_constant__ TmapSet mapV,
                   const __grid_constant__ TmapSet mapQ, const __grid_constant__ TmapSet mapO,
                   const GlobalProjArgs p) {
    extern __shared__ uint8_t smraw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int G = p.G, n = p.n, nch = (G + kGC - 1) / kGC;
    uint8_t *kbuf = base;                    // K tile; the V tile follows at +kTile16
    uint8_t *vbuf = kbuf + kTile16;
    uint8_t *qbuf = vbuf + kTile16;          // [nch] Qg chunks, 16 rows x 128 B
    uint8_t *obuf = qbuf + nch * 2048;       // [nch] dOg chunks
    uint8_t *pa = obuf + nch * 2048;         // P  [128 keys][16 queries], 128-B swizzled rows
    uint8_t *dsa = pa + kTile16;             // dS [128 keys][16 queries]
    uint8_t *dsb = dsa + kTile16;            // dS [16 queries][128 keys]: two 64-key blocks
    float *lse2 = reinterpret_cast<float *>(dsb + 2 * 2048);   // [256] lse * log2e
    float *del = lse2 + 256;                                    // [256] delta
    uint64_t *bars = reinterpret_cast<uint64_t *>(del + 256);
    uint64_t *ldfull = bars, *sfull = bars + 1, *pfull = bars + 2, *qfull = bars + 3, *qdone = bars + 4;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 6);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(tmem_holder + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt = blockIdx.x, bh = blockIdx.y, j0 = kt * kTcKeys;
    if (threadIdx.x == 0) {
        mbar_init(ldfull, 1);
        mbar_init(sfull, 1);
        mbar_init(pfull, 128);
        mbar_init(qfull, 1);
        mbar_init(qdone, 128);
        mbar_init(qdone + 1, 1);   // every product complete
        *abort_flag = 0;
        *no_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTcTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        // ---------------- loads: the key tile and every query chunk, once ----------------
        if (lane == 0) {
            mbar_arrive_expect_tx(ldfull, 2 * kTile16 + 2 * nch * 2048);
            tma_load_3d(kbuf, &mapK.m[0], ldfull, 0, j0, bh);
            tma_load_3d(vbuf, &mapV.m[0], ldfull, 0, j0, bh);
            for (int c = 0; c < nch; ++c) {
                tma_load_3d(qbuf + c * 2048, &mapQ.m[0], ldfull, 0, c * kGC, bh);
                tma_load_3d(obuf + c * 2048, &mapO.m[0], ldfull, 0, c * kGC, bh);
            }
        }
        __syncwarp();
        // the copies land before the CTA may exit
        mbar_wait(ldfull, 0, no_abort, nullptr, 100000000ull);
    } else if (warp == 1) {
        // ---------------- products (lane 0 issues) ----------------
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        constexpr uint32_t id_s = idesc_f16(kTcKeys, kGC, kBf16, false, false);   // S^T, dP^T
        constexpr uint32_t id_g = idesc_f16(kTcKeys, 64, kBf16, false, true);     // dV, dK
        constexpr uint32_t id_q = idesc_f16(kTcKeys, kGC, kBf16, true, false);    // dQ^T
        const uint64_t d_k = sdesc_sw128(smem_u32(kbuf), 16, 1024);
        const uint64_t d_v = sdesc_sw128(smem_u32(vbuf), 16, 1024);
        const uint64_t d_kmn = sdesc_sw128(smem_u32(kbuf), kTile16, 1024);   // K^T, MN-major A
        const uint64_t d_pa = sdesc_sw128(smem_u32(pa), 16, 1024);
        const uint64_t d_dsa = sdesc_sw128(smem_u32(dsa), 16, 1024);
        const uint64_t d_dsb = sdesc_sw128(smem_u32(dsb), 16, 1024);
        ok = __all_sync(0xffffffffu, mbar_wait(ldfull, 0, abort_flag, p.err));
        for (int c = 0; c < nch && ok; ++c) {
            if (c > 0 && !__all_sync(0xffffffffu, mbar_wait(qdone, (c - 1) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t qoff = (uint64_t)((c * 2048) >> 4);
            const uint64_t d_q = sdesc_sw128(smem_u32(qbuf), 16, 1024) + qoff;
            const uint64_t d_o = sdesc_sw128(smem_u32(obuf), 16, 1024) + qoff;
            const uint64_t d_qmn = sdesc_sw128(smem_u32(qbuf), 1024, 1024) + qoff;
            const uint64_t d_omn = sdesc_sw128(smem_u32(obuf), 1024, 1024) + qoff;
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    mma_f16_ss(tmem + kColS, d_k + 2 * k, d_q + 2 * k, id_s, k > 0 ? 1u : 0u);
                    mma_f16_ss(tmem + kColDP, d_v + 2 * k, d_o + 2 * k, id_s, k > 0 ? 1u : 0u);
                }
                mma_commit(sfull);
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(pfull, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                mma_f16_ss(tmem + kColDV, d_pa, d_omn, id_g, c > 0 ? 1u : 0u);
                mma_f16_ss(tmem + kColDK, d_dsa, d_qmn, id_g, c > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < kTcKeys / 16; ++k) {
                    const uint64_t a = d_kmn + (uint64_t)((2048 * k) >> 4);
                    const uint64_t b = d_dsb + (uint64_t)((((k >> 2) * 2048) + (k & 3) * 32) >> 4);
                    mma_f16_ss(tmem + kColDQ, a, b, id_q, k > 0 ? 1u : 0u);
                }
                mma_commit(qfull);
            }
            __syncwarp();
        }
        // the products issued complete before tensor memory is freed
        if (lane == 0) mma_commit(qdone + 1);
        __syncwarp();
    } else {
        // ---------------- workers: lane = key m of the tile ----------------
        const int quarter = warp & 3, m = quarter * 32 + lane, t = threadIdx.x - 64;
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        const T *Og = reinterpret_cast<const T *>(p.Og) + (long long)bh * G * 64;
        const T *dOg = reinterpret_cast<const T *>(p.dOg) + (long long)bh * G * 64;
        for (int gg = t; gg < G; gg += 128) {
            lse2[gg] = *GP(p.bnd, p.lseg + (long long)bh * G + gg) * kLog2e;
            float d = 0.f;
            for (int c = 0; c < 64; ++c)
                d = fmaf(Elt<T>::to_f(*GP(p.bnd, Og + (long long)gg * 64 + c)),
                         Elt<T>::to_f(*GP(p.bnd, dOg + (long long)gg * 64 + c)), d);
            del[gg] = d;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");   // the workers' lse, delta
        const bool kvalid = j0 + m < n;
        const float xs = p.scale * kLog2e;
        // this key's bias (log2 units), the same for every global query
        const float kb = (p.kbias && kvalid) ? *GP(p.bnd, p.kbias + (size_t)(bh / p.h) * n + j0 + m) * kLog2e : 0.f;
        const uint32_t pa_row = smem_u32(pa) + m * 128, dsa_row = smem_u32(dsa) + m * 128;
        for (int c = 0; c < nch && ok; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait(sfull, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[16], dv[16];
            tmem_ld16(lane_base + kColS, sv);
            tmem_ld16(lane_base + kColDP, dv);
            tmem_ld_wait();
            float pv[16], dsv[16];
#pragma unroll
            for (int q = 0; q < kGC; ++q) {
                const int gg = c * kGC + q;
                const bool live = kvalid && gg < G;
                const float pr = live ? ex2(fmaf(__uint_as_float(sv[q]), xs, kb) - lse2[gg < G ? gg : 0]) : 0.f;
                pv[q] = pr;
                dsv[q] = pr * (__uint_as_float(dv[q]) - (gg < G ? del[gg] : 0.f));
            }
            // P and dS rows (queries 0-15 of the chunk: the first two 16-byte
            // pieces of the row, swizzled), and dS as [query][key]
            sts16(pa_row + ((0 ^ (m & 7)) << 4), make_uint4(pack2<T>(pv[0], pv[1]), pack2<T>(pv[2], pv[3]),
                                                            pack2<T>(pv[4], pv[5]), pack2<T>(pv[6], pv[7])));
            sts16(pa_row + ((1 ^ (m & 7)) << 4), make_uint4(pack2<T>(pv[8], pv[9]), pack2<T>(pv[10], pv[11]),
                                                            pack2<T>(pv[12], pv[13]), pack2<T>(pv[14], pv[15])));
            sts16(dsa_row + ((0 ^ (m & 7)) << 4), make_uint4(pack2<T>(dsv[0], dsv[1]), pack2<T>(dsv[2], dsv[3]),
                                                             pack2<T>(dsv[4], dsv[5]), pack2<T>(dsv[6], dsv[7])));
            sts16(dsa_row + ((1 ^ (m & 7)) << 4), make_uint4(pack2<T>(dsv[8], dsv[9]), pack2<T>(dsv[10], dsv[11]),
                                                             pack2<T>(dsv[12], dsv[13]), pack2<T>(dsv[14], dsv[15])));
            {
                uint16_t *blk = reinterpret_cast<uint16_t *>(dsb + (m >> 6) * 2048);
                const int col = m & 63;   // key within the 64-key block
#pragma unroll
                for (int q = 0; q < kGC; q += 2) {
                    const uint32_t w2 = pack2<T>(dsv[q], dsv[q + 1]);
                    blk[q * 64 + ((((col >> 3) ^ (q & 7))) << 3) + (col & 7)] = (uint16_t)(w2 & 0xffffu);
                    blk[(q + 1) * 64 + ((((col >> 3) ^ ((q + 1) & 7))) << 3) + (col & 7)] = (uint16_t)(w2 >> 16);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(pfull);
            if (!__all_sync(0xffffffffu, mbar_wait(qfull, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (quarter < 2) {   // TMEM lanes 0-63: the 64 channels of dQ^T
                uint32_t qv[16];
                tmem_ld16(lane_base + kColDQ, qv);
                tmem_ld_wait();
                float *part = p.ws + ((long long)bh * p.nchunks + kt) * G * 64 + m;
#pragma unroll
                for (int q = 0; q < kGC; ++q) {
                    const int gg = c * kGC + q;
                    if (gg < G) *GP(p.bnd, part + (long long)gg * 64) = p.scale * __uint_as_float(qv[q]);
                }
            }
            tc_fence_before();
            mbar_arrive(qdone);
        }
        // dV, dK rows of this key (the last chunk's products are complete)
        if (ok) {
            tc_fence_after();
            T *dV = reinterpret_cast<T *>(p.dVg) + ((long long)bh * n + j0 + m) * 64;
            T *dK = reinterpret_cast<T *>(p.dKg) + ((long long)bh * n + j0 + m) * 64;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const float mul = which ? p.scale : 1.f;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + (which ? kColDK : kColDV) + 32 * h, v);
                    tmem_ld_wait();
                    if (kvalid) {
                        uint4 *o4 = reinterpret_cast<uint4 *>((which ? dK : dV) + 32 * h);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            *GP(p.bnd, o4 + u) = make_uint4(
                                pack2<T>(mul * __uint_as_float(v[8 * u]), mul * __uint_as_float(v[8 * u + 1])),
                                pack2<T>(mul * __uint_as_float(v[8 * u + 2]), mul * __uint_as_float(v[8 * u + 3])),
                                pack2<T>(mul * __uint_as_float(v[8 * u + 4]), mul * __uint_as_float(v[8 * u + 5])),
                                pack2<T>(mul * __uint_as_float(v[8 * u + 6]), mul * __uint_as_float(v[8 * u + 7])));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        // every product issued has completed (its commit arrived) before the free
        mbar_wait(qdone + 1, 0, no_abort, nullptr, 100000000ull);
        __syncwarp();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

// ---------------------------------------------------------------------------
// forward on the tensor cores: CTA (128-key tile, slice), every global query
// in chunks of 16.  S^T = Kg Qg_c^T (M = 128 keys, N = 16); the workers (lane
// = key) take each query's max and sum over the tile's keys, write
// P = 2^(s - max) as [query][key], and O_c^T = Vg^T P (K = 128 keys; Vg read as
// an MN-major A of 128 rows whose second 64-row block is the K tile stored
// right after it: those output lanes are never read) gives the tile's
// unnormalised output.  The partial (max, sum,
// output) of every (slice, tile, query) goes to the workspace; the combine
// kernel merges the tiles.
// ---------------------------------------------------------------------------
constexpr uint32_t kFColS = 0, kFColO = 32;
constexpr uint32_t kFTmemCols = 64;   // S^T at columns 0-15, O^T at 32-47

__host__ __device__ constexpr int tc_fwd_smem(int nch) {
    return 1024 + 2 * kTile16 /* K, V */ + nch * 2048 /* Qg */ + 2 * 2048 /* P [query][key] */ +
           2 * 4 * kGC * 4 /* per-warp max, sum */ + 256;
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 4)
    k_gproj_fwd_tc(const __grid_constant__ TmapSet mapK, const __grid_constant__ TmapSet mapV,
                   const __grid_constant__ TmapSet mapQ, const GlobalProjArgs p) {
    extern __shared__ uint8_t smraw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int G = p.G, n = p.n, nch = (G + kGC - 1) / kGC;
    uint8_t *vbuf = base;                    // V tile; the K tile follows at +kTile16
    uint8_t *kbuf = vbuf + kTile16;
    uint8_t *qbuf = kbuf + kTile16;          // [nch] Qg chunks
    uint8_t *pb = qbuf + nch * 2048;         // P [16 queries][128 keys]: two 64-key blocks
    float *wmax = reinterpret_cast<float *>(pb + 2 * 2048);   // [4 warps][16]
    float *wsum = wmax + 4 * kGC;                               // [4 warps][16]
    uint64_t *bars = reinterpret_cast<uint64_t *>(wsum + 4 * kGC);
    uint64_t *ldfull = bars, *sfull = bars + 1, *pfull = bars + 2, *ofull = bars + 3, *odone = bars + 4,
             *alldone = bars + 5, *wbar = bars + 6;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 7);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(tmem_holder + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt = blockIdx.x, bh = blockIdx.y, j0 = kt * kTcKeys;
    if (threadIdx.x == 0) {
        mbar_init(ldfull, 1);
        mbar_init(sfull, 1);
        mbar_init(pfull, 128);
        mbar_init(ofull, 1);
        mbar_init(odone, 128);
        mbar_init(alldone, 1);
        mbar_init(wbar, 128);
        *abort_flag = 0;
        *no_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kFTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(ldfull, 2 * kTile16 + nch * 2048);
            tma_load_3d(kbuf, &mapK.m[0], ldfull, 0, j0, bh);
            tma_load_3d(vbuf, &mapV.m[0], ldfull, 0, j0, bh);
            for (int c = 0; c < nch; ++c) tma_load_3d(qbuf + c * 2048, &mapQ.m[0], ldfull, 0, c * kGC, bh);
        }
        __syncwarp();
        mbar_wait(ldfull, 0, no_abort, nullptr, 100000000ull);
    } else if (warp == 1) {
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        constexpr uint32_t id_s = idesc_f16(kTcKeys, kGC, kBf16, false, false);   // S^T
        constexpr uint32_t id_o = idesc_f16(kTcKeys, kGC, kBf16, true, false);    // O^T
        const uint64_t d_k = sdesc_sw128(smem_u32(kbuf), 16, 1024);
        const uint64_t d_vmn = sdesc_sw128(smem_u32(vbuf), kTile16, 1024);   // V^T, MN-major A
        const uint64_t d_pb = sdesc_sw128(smem_u32(pb), 16, 1024);
        ok = __all_sync(0xffffffffu, mbar_wait(ldfull, 0, abort_flag, p.err));
        for (int c = 0; c < nch && ok; ++c) {
            if (c > 0 && !__all_sync(0xffffffffu, mbar_wait(odone, (c - 1) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t d_q = sdesc_sw128(smem_u32(qbuf), 16, 1024) + (uint64_t)((c * 2048) >> 4);
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_f16_ss(tmem + kFColS, d_k + 2 * k, d_q + 2 * k, id_s, k > 0 ? 1u : 0u);
                mma_commit(sfull);
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(pfull, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kTcKeys / 16; ++k) {
                    const uint64_t a = d_vmn + (uint64_t)((2048 * k) >> 4);
                    const uint64_t b = d_pb + (uint64_t)((((k >> 2) * 2048) + (k & 3) * 32) >> 4);
                    mma_f16_ss(tmem + kFColO, a, b, id_o, k > 0 ? 1u : 0u);
                }
                mma_commit(ofull);
            }
            __syncwarp();
        }
        if (lane == 0) mma_commit(alldone);
        __syncwarp();
    } else {
        const int quarter = warp & 3, wi = warp - 2, m = quarter * 32 + lane, t = threadIdx.x - 64;
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        const bool kvalid = j0 + m < n;
        const float xs = p.scale * kLog2e;
        // the four worker warps meet on wbar (bounded waits, so a timeout
        // anywhere lets every warp leave); nb counts its phases
        uint32_t nb = 0;
        auto meet = [&]() -> bool {
            mbar_arrive(wbar);
            return __all_sync(0xffffffffu, mbar_wait(wbar, (nb++) & 1, abort_flag, p.err));
        };
        for (int c = 0; c < nch && ok; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait(sfull, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[16];
            tmem_ld16(lane_base + kFColS, sv);
            tmem_ld_wait();
            float x[16];
#pragma unroll
            for (int q = 0; q < kGC; ++q) x[q] = kvalid ? __uint_as_float(sv[q]) * xs : -INFINITY;
            // max over the tile's 128 keys of every query: warp, then the 4 warps
#pragma unroll
            for (int q = 0; q < kGC; ++q) {
                float v = x[q];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                if (lane == q) wmax[wi * kGC + q] = v;
            }
            if (!meet()) {
                ok = false;
                break;
            }
            float pr[16];
#pragma unroll
            for (int q = 0; q < kGC; ++q) {
                const float mx = max3(wmax[q], wmax[kGC + q], fmaxf(wmax[2 * kGC + q], wmax[3 * kGC + q]));
                pr[q] = ex2(x[q] - mx);   // 0 for keys past the end (the tile has one key < n)
            }
            // P as [query][key] (two 64-key blocks, 128-byte swizzled rows)
            {
                uint16_t *blk = reinterpret_cast<uint16_t *>(pb + (m >> 6) * 2048);
                const int col = m & 63;
#pragma unroll
                for (int q = 0; q < kGC; q += 2) {
                    const uint32_t w2 = pack2<T>(pr[q], pr[q + 1]);
                    blk[q * 64 + ((((col >> 3) ^ (q & 7))) << 3) + (col & 7)] = (uint16_t)(w2 & 0xffffu);
                    blk[(q + 1) * 64 + ((((col >> 3) ^ ((q + 1) & 7))) << 3) + (col & 7)] = (uint16_t)(w2 >> 16);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(pfull);
            // sums over the keys (of the fp32 values; the product uses them rounded)
#pragma unroll
            for (int q = 0; q < kGC; ++q) {
                float v = pr[q];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == q) wsum[wi * kGC + q] = v;
            }
            if (!meet()) {
                ok = false;
                break;
            }
            // the partial of (slice, tile, query): [max (log2 units), sum, O[64]]
            float *part = p.ws + ((long long)bh * p.nchunks + kt) * G * 66;
            if (t < kGC && c * kGC + t < G) {
                const int gg = c * kGC + t;
                *GP(p.bnd, part + (long long)gg * 66) =
                    max3(wmax[t], wmax[kGC + t], fmaxf(wmax[2 * kGC + t], wmax[3 * kGC + t]));
                *GP(p.bnd, part + (long long)gg * 66 + 1) =
                    (wsum[t] + wsum[kGC + t]) + (wsum[2 * kGC + t] + wsum[3 * kGC + t]);
            }
            if (!__all_sync(0xffffffffu, mbar_wait(ofull, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (quarter < 2) {   // TMEM lanes 0-63: the 64 channels of O^T
                uint32_t ov[16];
                tmem_ld16(lane_base + kFColO, ov);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < kGC; ++q) {
                    const int gg = c * kGC + q;
                    if (gg < G) *GP(p.bnd, part + (long long)gg * 66 + 2 + m) = __uint_as_float(ov[q]);
                }
            }
            tc_fence_before();
            // the next chunk's maxima and sums overwrite these slots
            if (!meet()) {
                ok = false;
                break;
            }
            mbar_arrive(odone);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        mbar_wait(alldone, 0, no_abort, nullptr, 100000000ull);
        __syncwarp();
        tmem_dealloc(tmem, kFTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Global columns of the fused forward with global tokens, on the tensor
// cores (G <= 64): CTA per (128-query tile, slice).  S = Q_tile K_G^T
// (N = G rounded up to 16), each worker lane owns a query row and takes the
// softmax over the global keys in registers, O_B = P V_G (K = G rounded up),
// and the row's (O_B, lse_B) is merged into the band part's (O, lse) by
// log-sum-exp.  The Q tile arrives by TMA; the few K_G, V_G rows are loaded
// by warp 0 and written into the swizzled layout (zeros past G).  Rows in G
// are left to the dense rows.
// ---------------------------------------------------------------------------
constexpr uint32_t kCColS = 0, kCColO = 64;
constexpr uint32_t kCTmemCols = 128;

__host__ __device__ constexpr int tc_cols_smem() {
    return 1024 + kTile16 /* Q tile */ + 2 * 64 * 128 /* K_G, V_G: 64 rows */ + kTile16 /* P */ + 128;
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 3)   // three CTAs an SM (tensor memory allows four)
    k_fused_glob_cols_tc(const __grid_constant__ TmapSet mapQ, const GlobalRowsArgs p) {
    extern __shared__ uint8_t smraw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int G = p.gl.G, n = p.n, gp = (G + 15) & ~15;   // global keys, rounded up to 16
    uint8_t *qbuf = base;                    // Q tile [128 x 64]
    uint8_t *kgb = qbuf + kTile16;           // K_G [gp rows x 64]
    uint8_t *vgb = kgb + 64 * 128;           // V_G [gp rows x 64]
    uint8_t *pa = vgb + 64 * 128;            // P [128 queries][gp keys], 128-byte swizzled rows
    uint64_t *bars = reinterpret_cast<uint64_t *>(pa + kTile16);
    uint64_t *ldfull = bars, *sfull = bars + 1, *pfull = bars + 2, *ofull = bars + 3;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(tmem_holder + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, bh = blockIdx.y, a0 = qt * kTcKeys;
    // the key bias of the global keys (log2 units; 0 past G), visible to the
    // workers after the block barrier below
    __shared__ __align__(16) float gbias[64];
    if (p.kbias && threadIdx.x < 64)
        gbias[threadIdx.x] =
            threadIdx.x < G ? *GP(p.bnd, p.kbias + (size_t)(bh / p.h) * n + p.gl.idx[threadIdx.x]) * kLog2e : 0.f;
    if (threadIdx.x == 0) {
        mbar_init(ldfull, 1 + 32);   // the Q copy, and warp 0's lanes after K_G, V_G
        mbar_init(sfull, 1);
        mbar_init(pfull, 128);
        mbar_init(ofull, 1);
        *abort_flag = 0;
        *no_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kCTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(ldfull, kTile16);
            tma_load_3d(qbuf, &mapQ.m[0], ldfull, 0, a0, bh);
        }
        // K_G, V_G rows (zeros past G) written straight into the 128-byte
        // swizzled layout: 16-byte piece c of row r at r * 128 + ((c ^ (r & 7)) << 4)
        const T *Kb = reinterpret_cast<const T *>(p.K) + (long long)bh * n * 64;
        const T *Vb = reinterpret_cast<const T *>(p.V) + (long long)bh * n * 64;
        for (int e = lane; e < gp * 8; e += 32) {
            const int r = e >> 3, c = e & 7;
            uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
            if (r < G) {
                kv = ldg16(GPN(p.bnd, Kb + (long long)p.gl.idx[r] * 64 + 8 * c, 16));
                vv = ldg16(GPN(p.bnd, Vb + (long long)p.gl.idx[r] * 64 + 8 * c, 16));
            }
            const uint32_t off = r * 128 + ((c ^ (r & 7)) << 4);
            sts16(smem_u32(kgb) + off, kv);
            sts16(smem_u32(vgb) + off, vv);
        }
        fence_proxy_async_smem();
        mbar_arrive(ldfull);
        mbar_wait(ldfull, 0, no_abort, nullptr, 100000000ull);
    } else if (warp == 1) {
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        const uint32_t id_s = idesc_f16(kTcKeys, gp, kBf16, false, false);
        constexpr uint32_t id_o = idesc_f16(kTcKeys, 64, kBf16, false, true);
        const uint64_t d_q = sdesc_sw128(smem_u32(qbuf), 16, 1024);
        const uint64_t d_kg = sdesc_sw128(smem_u32(kgb), 16, 1024);
        const uint64_t d_vmn = sdesc_sw128(smem_u32(vgb), 1024, 1024);   // V_G as MN-major B
        const uint64_t d_pa = sdesc_sw128(smem_u32(pa), 16, 1024);
        ok = __all_sync(0xffffffffu, mbar_wait(ldfull, 0, abort_flag, p.err));
        if (ok) {
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_f16_ss(tmem + kCColS, d_q + 2 * k, d_kg + 2 * k, id_s, k > 0 ? 1u : 0u);
                mma_commit(sfull);
            }
            __syncwarp();
            ok = __all_sync(0xffffffffu, mbar_wait(pfull, 0, abort_flag, p.err));
        }
        if (ok) {
            tc_fence_after();
            if (lane == 0) {
                for (int k = 0; k < gp / 16; ++k)
                    mma_f16_ss(tmem + kCColO, d_pa + 2 * k, d_vmn + (uint64_t)((2048 * k) >> 4), id_o, k > 0 ? 1u : 0u);
                mma_commit(ofull);
            }
            __syncwarp();
        } else if (lane == 0) {
            mma_commit(ofull);   // the products issued complete before the free
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3, m = quarter * 32 + lane;
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        const int i = a0 + m;
        bool write = i < n;
        if (write) {
            int lo = 0, hi = G;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (p.gl.idx[mid] < i) lo = mid + 1; else hi = mid;
            }
            write = !(lo < G && p.gl.idx[lo] == i);
        }
        const float xs = p.scale * kLog2e;
        float mb = 0.f, lb = 1.f;
        if (__all_sync(0xffffffffu, mbar_wait(sfull, 0, abort_flag, p.err))) {
            tc_fence_after();
            // every index compile-time (registers), the columns past gp unused
            float x[64];
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                if (c0 < gp) {   // warp-uniform
                    uint32_t v[16];
                    tmem_ld16(lane_base + kCColS + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) x[c0 + u] = __uint_as_float(v[u]);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) x[c0 + u] = 0.f;
                }
            }
            mb = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) x[c] = c < G ? x[c] * xs : -INFINITY;
            if (p.kbias) {   // the key bias of global key c (staged above), the same for every row
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 kb = *reinterpret_cast<const float4 *>(&gbias[c]);
                    x[c] += kb.x;
                    x[c + 1] += kb.y;
                    x[c + 2] += kb.z;
                    x[c + 3] += kb.w;
                }
            }
#pragma unroll
            for (int c = 0; c < 64; ++c) mb = fmaxf(mb, x[c]);
            lb = 0.f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                x[c] = ex2(x[c] - mb);   // 0 past G
                lb += x[c];
            }
            // P row m: keys 0..gp-1 = the first gp / 8 swizzled 16-byte pieces
            const uint32_t prow = smem_u32(pa) + m * 128;
#pragma unroll
            for (int c = 0; c < 64; c += 8)
                if (c < gp)
                    sts16(prow + ((((c >> 3)) ^ (m & 7)) << 4),
                          make_uint4(pack2<T>(x[c], x[c + 1]), pack2<T>(x[c + 2], x[c + 3]),
                                     pack2<T>(x[c + 4], x[c + 5]), pack2<T>(x[c + 6], x[c + 7])));
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(pfull);
        } else {
            ok = false;
        }
        if (ok && __all_sync(0xffffffffu, mbar_wait(ofull, 0, abort_flag, p.err))) {
            tc_fence_after();
            uint32_t ov[32];
            const long long row = (long long)bh * n + (write ? i : 0);
            const float lse_a = write ? *GP(p.bnd, p.lse + row) : 0.f;
            const float lse_b = mb / kLog2e + logf(lb);
            const float m2 = fmaxf(lse_a, lse_b);
            const float wa = expf(lse_a - m2), wb = expf(lse_b - m2);
            const float den = wa + wb;
            const float fa = wa / den, fb = wb / (lb * den);
            uint4 *o4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.O) + row * 64);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                tmem_ld32(lane_base + kCColO + 32 * h, ov);
                tmem_ld_wait();
                if (write) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 a = *GP(p.bnd, o4 + 4 * h + k);
                        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
                        uint32_t r[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int c = 8 * k + 2 * u;
                            r[u] = pack2<T>(fmaf(lo16<T>(w[u]), fa, __uint_as_float(ov[c]) * fb),
                                            fmaf(hi16<T>(w[u]), fa, __uint_as_float(ov[c + 1]) * fb));
                        }
                        *GP(p.bnd, o4 + 4 * h + k) = make_uint4(r[0], r[1], r[2], r[3]);
                    }
                }
            }
            if (write) *GP(p.bnd, p.lse + row) = m2 + logf(den);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        mbar_wait(ofull, 0, no_abort, nullptr, 100000000ull);
        __syncwarp();
        tmem_dealloc(tmem, kCTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Dense global rows of the fused forward on the tensor cores: CTA per (16
// global queries, slice) over every key, no workspace.  As in the global
// projections the keys are the M side: S^T = K_c Q^T gives each worker lane
// one key with the 16 queries' scores in its columns.  Pass 1 walks the
// 128-key chunks for every query's maximum; pass 2 recomputes S^T, forms
// P = 2^(s - max) and accumulates O^T += V_c^T P^T in tensor memory while each
// lane sums its keys' P.  The maximum is final before pass 2, so nothing is
// rescaled, and the sums are merged once at the end.  K (pass 1) or K and V
// (pass 2) chunks arrive by TMA through a four-stage ring; S^T and P are
// double-buffered so a chunk's softmax overlaps the next chunk's product.
// ---------------------------------------------------------------------------
constexpr int kRStages = 4;
constexpr uint32_t kRColS = 0, kRColO = 32;   // S^T buffers at columns 0 and 16, O^T at 32
constexpr uint32_t kRTmemCols = 64;

__host__ __device__ constexpr int tc_rows_smem() {
    return 1024 + kRStages * 2 * kTile16 /* V, K ring */ + 2048 /* Q */ + 2 * 4096 /* P */ +
           2 * 4 * kGC * 4 /* per-warp max, sum */ + 256;
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_fused_glob_rows_tc(const __grid_constant__ TmapSet mapK, const __grid_constant__ TmapSet mapV,
                         const GlobalRowsArgs p) {
    extern __shared__ uint8_t smraw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const int G = p.gl.G, n = p.n, nck = (n + kTcKeys - 1) / kTcKeys, steps = 2 * nck;
    uint8_t *ring = base;                            // stage b: V at +0, K at +kTile16
    uint8_t *qbuf = ring + kRStages * 2 * kTile16;   // Q [16 queries][64]
    uint8_t *pbuf = qbuf + 2048;                     // two P [16 queries][128 keys]
    float *wmax = reinterpret_cast<float *>(pbuf + 2 * 4096);   // [4 warps][16]
    float *wsum = wmax + 4 * kGC;                                // [4 warps][16]
    uint64_t *bars = reinterpret_cast<uint64_t *>(wsum + 4 * kGC);
    uint64_t *kvfull = bars, *kvempty = bars + kRStages, *sfull = bars + 2 * kRStages, *sempty = sfull + 2,
             *pfull = sempty + 2, *pempty = pfull + 2, *ofull = pempty + 2, *red = ofull + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(red + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(tmem_holder + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gc = blockIdx.x, bh = blockIdx.y;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRStages; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], 128);
            mbar_init(&pfull[i], 128);
            mbar_init(&pempty[i], 1);
        }
        mbar_init(ofull, 1);
        mbar_init(red, 128);
        *abort_flag = 0;
        *no_abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x >= 64) {
        // the 16 queries' rows into the swizzled Q tile, zeros past G
        const int t = threadIdx.x - 64, j = t >> 3, c = t & 7, gg = gc * kGC + j;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (gg < G) v = ldg16(GPN(p.bnd, reinterpret_cast<const T *>(p.Q) + ((long long)bh * n + p.gl.idx[gg]) * 64 + 8 * c, 16));
        sts16(smem_u32(qbuf) + j * 128 + ((c ^ (j & 7)) << 4), v);
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kRTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    bool ok = true;

    if (warp == 0) {
        int issued = 0;
        for (int st = 0; st < steps && ok; ++st) {
            const int b = st % kRStages, c = st < nck ? st : st - nck;
            if (!__all_sync(0xffffffffu, mbar_wait(&kvempty[b], ((st / kRStages) & 1) ^ 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                uint8_t *stage = ring + b * 2 * kTile16;
                mbar_arrive_expect_tx(&kvfull[b], st < nck ? kTile16 : 2 * kTile16);
                tma_load_3d(stage + kTile16, &mapK.m[0], &kvfull[b], 0, c * kTcKeys, bh);
                if (st >= nck) tma_load_3d(stage, &mapV.m[0], &kvfull[b], 0, c * kTcKeys, bh);
            }
            __syncwarp();
            ++issued;
        }
        // the copies still in flight land before the CTA ends
        for (int k = issued > kRStages ? issued - kRStages : 0; k < issued; ++k)
            mbar_wait(&kvfull[k % kRStages], (k / kRStages) & 1, no_abort, nullptr, 100000000ull);
    } else if (warp == 1) {
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        constexpr uint32_t id_s = idesc_f16(kTcKeys, kGC, kBf16, false, false);   // S^T = K Q^T
        constexpr uint32_t id_o = idesc_f16(kTcKeys, kGC, kBf16, true, false);    // O^T += V^T P^T
        const uint64_t d_q = sdesc_sw128(smem_u32(qbuf), 16, 1024);
        const uint64_t d_k = sdesc_sw128(smem_u32(ring + kTile16), 16, 1024);
        // V^T as an MN-major A of 128 rows: its second 64-row block is the
        // stage's K tile, and those output lanes are never read
        const uint64_t d_vmn = sdesc_sw128(smem_u32(ring), kTile16, 1024);
        const uint64_t d_p = sdesc_sw128(smem_u32(pbuf), 16, 1024);
        // O^T += V_c^T P_c^T for the pass-2 step u, once its P is written
        auto pv = [&](int u) -> bool {
            const int c2 = u - nck, pi = c2 & 1, bu = u % kRStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&pfull[pi], (c2 >> 1) & 1, abort_flag, p.err))) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t voff = (uint64_t)((bu * 2 * kTile16) >> 4);
#pragma unroll
                for (int k = 0; k < kTcKeys / 16; ++k) {
                    const uint64_t a = d_vmn + voff + (uint64_t)((2048 * k) >> 4);
                    const uint64_t b = d_p + (uint64_t)((pi * 4096 + (k >> 2) * 2048 + (k & 3) * 32) >> 4);
                    mma_f16_ss(tmem + kRColO, a, b, id_o, (c2 > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&pempty[pi]);
                mma_commit(&kvempty[bu]);
            }
            __syncwarp();
            return true;
        };
        for (int st = 0; st < steps && ok; ++st) {
            const int b = st % kRStages, sb = st & 1;
            bool w = mbar_wait(&kvfull[b], (st / kRStages) & 1, abort_flag, p.err);
            w = w && mbar_wait(&sempty[sb], ((st >> 1) & 1) ^ 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint64_t koff = (uint64_t)((b * 2 * kTile16) >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16_ss(tmem + kRColS + 16 * sb, d_k + koff + 2 * k, d_q + 2 * k, id_s, k > 0 ? 1u : 0u);
                mma_commit(&sfull[sb]);
                if (st < nck) mma_commit(&kvempty[b]);   // pass 1 needs only K
            }
            __syncwarp();
            // the previous chunk's product, issued after this one's scores
            if (st > nck && !pv(st - 1)) ok = false;
        }
        if (ok && !pv(steps - 1)) ok = false;
        if (lane == 0) mma_commit(ofull);   // also: every product issued is complete
        __syncwarp();
    } else {
        const int quarter = warp & 3, wi = warp - 2, m = quarter * 32 + lane;
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        const float xs = p.scale * kLog2e;
        float mx[kGC], ls[kGC];
#pragma unroll
        for (int q = 0; q < kGC; ++q) {
            mx[q] = -INFINITY;
            ls[q] = 0.f;
        }
        for (int st = 0; st < steps && ok; ++st) {
            const int sb = st & 1, c = st < nck ? st : st - nck;
            if (!__all_sync(0xffffffffu, mbar_wait(&sfull[sb], (st >> 1) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[16];
            tmem_ld16(lane_base + kRColS + 16 * sb, sv);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&sempty[sb]);   // the scores are in registers
            const bool kvalid = c * kTcKeys + m < n;
            // this key's bias (log2 units), the same for the chunk's 16 queries
            const float kb = (p.kbias && kvalid)
                                 ? *GP(p.bnd, p.kbias + (size_t)(bh / p.h) * n + c * kTcKeys + m) * kLog2e
                                 : 0.f;
            if (st < nck) {
                if (kvalid) {
#pragma unroll
                    for (int q = 0; q < kGC; ++q) mx[q] = fmaxf(mx[q], fmaf(__uint_as_float(sv[q]), xs, kb));
                }
                if (st == nck - 1) {
                    // every query's maximum: the warp's keys, then the four warps
#pragma unroll
                    for (int q = 0; q < kGC; ++q) {
                        float v = mx[q];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                        if (lane == q) wmax[wi * kGC + q] = v;
                    }
                    mbar_arrive(red);
                    if (!__all_sync(0xffffffffu, mbar_wait(red, 0, abort_flag, p.err))) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int q = 0; q < kGC; ++q)
                        mx[q] = max3(wmax[q], wmax[kGC + q], fmaxf(wmax[2 * kGC + q], wmax[3 * kGC + q]));
                }
            } else {
                const int c2 = st - nck, pi = c2 & 1;
                float pr[kGC];
#pragma unroll
                for (int q = 0; q < kGC; ++q) {
                    pr[q] = kvalid ? ex2(fmaf(__uint_as_float(sv[q]), xs, kb) - mx[q]) : 0.f;
                    ls[q] += pr[q];
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&pempty[pi], ((c2 >> 1) & 1) ^ 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                // key m's column of P [query][key] (two 64-key blocks, 128-byte swizzled rows)
                uint16_t *blk = reinterpret_cast<uint16_t *>(pbuf + pi * 4096 + (m >> 6) * 2048);
                const int col = m & 63;
#pragma unroll
                for (int q = 0; q < kGC; q += 2) {
                    const uint32_t w2 = pack2<T>(pr[q], pr[q + 1]);
                    blk[q * 64 + (((col >> 3) ^ (q & 7)) << 3) + (col & 7)] = (uint16_t)(w2 & 0xffffu);
                    blk[(q + 1) * 64 + (((col >> 3) ^ ((q + 1) & 7)) << 3) + (col & 7)] = (uint16_t)(w2 >> 16);
                }
                fence_proxy_async_smem();
                mbar_arrive(&pfull[pi]);
            }
        }
        if (ok) {
            // every query's sum over the keys: the warp's lanes, then the four warps
#pragma unroll
            for (int q = 0; q < kGC; ++q) {
                float v = ls[q];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == q) wsum[wi * kGC + q] = v;
            }
            mbar_arrive(red);
            ok = __all_sync(0xffffffffu, mbar_wait(red, 1, abort_flag, p.err));
        }
        if (ok && __all_sync(0xffffffffu, mbar_wait(ofull, 0, abort_flag, p.err))) {
            tc_fence_after();
            float inv[kGC];
#pragma unroll
            for (int q = 0; q < kGC; ++q) {
                const float l = (wsum[q] + wsum[kGC + q]) + (wsum[2 * kGC + q] + wsum[3 * kGC + q]);
                inv[q] = 1.f / l;
                const int gg = gc * kGC + q;
                if (wi == 0 && lane == q && gg < G)
                    *GP(p.bnd, p.lse + (long long)bh * n + p.gl.idx[gg]) = mx[q] / kLog2e + logf(l);
            }
            if (quarter < 2) {   // TMEM lanes 0-63: the 64 channels of O^T
                uint32_t ov[16];
                tmem_ld16(lane_base + kRColO, ov);
                tmem_ld_wait();
                T *O = reinterpret_cast<T *>(p.O);
#pragma unroll
                for (int q = 0; q < kGC; ++q) {
                    const int gg = gc * kGC + q;
                    if (gg < G)
                        *GP(p.bnd, O + ((long long)bh * n + p.gl.idx[gg]) * 64 + m) = Elt<T>::from_f(__uint_as_float(ov[q]) * inv[q]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        mbar_wait(ofull, 0, no_abort, nullptr, 100000000ull);
        __syncwarp();
        tmem_dealloc(tmem, kRTmemCols);
    }
}

// dQg = sum of the key tiles' partials (fixed order): a thread per (slice,
// query, channel), eight loads in flight
template <typename T>
__global__ void __launch_bounds__(kThreads) k_gproj_dq(const GlobalProjArgs p) {
    const long long e = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (e >= (long long)p.BH * p.G * 64) return;
    const int c = (int)(e & 63);
    const long long bg = e >> 6, bh = bg / p.G, gg = bg - bh * p.G;
    const float *base = p.ws + ((long long)bh * p.nchunks * p.G + gg) * 64 + c;
    const long long step = (long long)p.G * 64;
    float s = 0.f;
    int k = 0;
    for (; k + 8 <= p.nchunks; k += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = *GP(p.bnd, base + (k + u) * step);
#pragma unroll
        for (int u = 0; u < 8; ++u) s += v[u];
    }
    for (; k < p.nchunks; ++k) s += *GP(p.bnd, base + k * step);
    *GP(p.bnd, reinterpret_cast<T *>(p.dQg) + e) = Elt<T>::from_f(s);
}

template <typename T>
cudaError_t launch_fwd_t(GlobalProjArgs a, cudaStream_t st) {
    a.nchunks = (a.n + kChunkKeys - 1) / kChunkKeys;
    const dim3 grid(a.nchunks, (a.G + kGC - 1) / kGC, a.BH);
    k_gproj_fwd<T><<<grid, kThreads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long warps = (long long)a.BH * a.G;
    const long long per_block = kThreads / 32;
    k_gproj_combine<T><<<(unsigned)((warps + per_block - 1) / per_block), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd_tc_t(const TmapSet &mk, const TmapSet &mv, const TmapSet &mq, GlobalProjArgs a,
                            cudaStream_t st) {
    a.nchunks = (a.n + kTcKeys - 1) / kTcKeys;
    const int nch = (a.G + kGC - 1) / kGC;
    const size_t smem = (size_t)tc_fwd_smem(nch);   // up to four CTAs per SM (64 TMEM columns each)
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gproj_fwd_tc<T>), smem);
    if (e != cudaSuccess) return e;
    k_gproj_fwd_tc<T><<<dim3(a.nchunks, a.BH), kTcThreads, smem, st>>>(mk, mv, mq, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long warps = (long long)a.BH * a.G;
    const long long per_block = kThreads / 32;
    k_gproj_combine<T><<<(unsigned)((warps + per_block - 1) / per_block), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_tc_t(const TmapSet &mk, const TmapSet &mv, const TmapSet &mq, const TmapSet &mo,
                            GlobalProjArgs a, cudaStream_t st) {
    a.nchunks = (a.n + kTcKeys - 1) / kTcKeys;
    const int nch = (a.G + kGC - 1) / kGC;
    // at least 80 KB: two CTAs per SM, as many as tensor memory holds (256 columns each)
    const size_t smem = (size_t)max(tc_bwd_smem(nch), 80 * 1024);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gproj_bwd_tc<T>), smem);
    if (e != cudaSuccess) return e;
    k_gproj_bwd_tc<T><<<dim3(a.nchunks, a.BH), kTcThreads, smem, st>>>(mk, mv, mq, mo, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long outs = (long long)a.BH * a.G * 64;
    k_gproj_dq<T><<<(unsigned)((outs + kThreads - 1) / kThreads), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_t(GlobalProjArgs a, cudaStream_t st) {
    a.nchunks = (a.n + kKT - 1) / kKT;
    const dim3 grid(a.nchunks, a.BH);
    const size_t smem = kBwdSmemFloats * sizeof(float);
    cudaError_t e0 = ensure_smem(reinterpret_cast<const void *>(k_gproj_bwd<T>), smem);
    if (e0 != cudaSuccess) return e0;
    k_gproj_bwd<T><<<grid, kThreads, smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long outs = (long long)a.BH * a.G * 64;
    k_gproj_dq<T><<<(unsigned)((outs + kThreads - 1) / kThreads), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t global_proj_workspace_bytes(long long BH, int G, int n) {
    // forward partials per 128-key tile (tensor cores) or 256-key chunk (FFMA)
    const size_t fwd = (size_t)BH * ((n + kTcKeys - 1) / kTcKeys) * G * 66 * sizeof(float);
    const size_t bwd = (size_t)BH * ((n + kKT - 1) / kKT) * G * 64 * sizeof(float);
    return fwd > bwd ? fwd : bwd;
}

cudaError_t launch_global_proj_bwd_tc(DType dt, const TmapSet &mk, const TmapSet &mv, const TmapSet &mq,
                                      const TmapSet &mo, const GlobalProjArgs &a, cudaStream_t st) {
    if (a.BH > 65535 || a.G > 256) return cudaErrorInvalidValue;
    if (dt == kF16) return launch_bwd_tc_t<__half>(mk, mv, mq, mo, a, st);
    if (dt == kBF16) return launch_bwd_tc_t<__nv_bfloat16>(mk, mv, mq, mo, a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_global_proj_fwd_tc(DType dt, const TmapSet &mk, const TmapSet &mv, const TmapSet &mq,
                                      const GlobalProjArgs &a, cudaStream_t st) {
    if (a.BH > 65535 || a.G > 256) return cudaErrorInvalidValue;
    if (dt == kF16) return launch_fwd_tc_t<__half>(mk, mv, mq, a, st);
    if (dt == kBF16) return launch_fwd_tc_t<__nv_bfloat16>(mk, mv, mq, a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fused_glob_cols_tc(DType dt, const TmapSet &mq, const GlobalRowsArgs &a, cudaStream_t st) {
    if (a.gl.G > 64 || a.BH > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((a.n + kTcKeys - 1) / kTcKeys), (unsigned)a.BH);
    const size_t smem = (size_t)tc_cols_smem();
    cudaError_t e;
    if (dt == kF16) {
        e = ensure_smem(reinterpret_cast<const void *>(k_fused_glob_cols_tc<__half>), smem);
        if (e != cudaSuccess) return e;
        k_fused_glob_cols_tc<__half><<<grid, kTcThreads, smem, st>>>(mq, a);
    } else if (dt == kBF16) {
        e = ensure_smem(reinterpret_cast<const void *>(k_fused_glob_cols_tc<__nv_bfloat16>), smem);
        if (e != cudaSuccess) return e;
        k_fused_glob_cols_tc<__nv_bfloat16><<<grid, kTcThreads, smem, st>>>(mq, a);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_fused_glob_rows_tc(DType dt, const TmapSet &mk, const TmapSet &mv, const GlobalRowsArgs &a,
                                      cudaStream_t st) {
    if (a.BH > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((a.gl.G + kGC - 1) / kGC), (unsigned)a.BH);
    const size_t smem = (size_t)tc_rows_smem();
    cudaError_t e;
    if (dt == kF16) {
        e = ensure_smem(reinterpret_cast<const void *>(k_fused_glob_rows_tc<__half>), smem);
        if (e != cudaSuccess) return e;
        k_fused_glob_rows_tc<__half><<<grid, kTcThreads, smem, st>>>(mk, mv, a);
    } else if (dt == kBF16) {
        e = ensure_smem(reinterpret_cast<const void *>(k_fused_glob_rows_tc<__nv_bfloat16>), smem);
        if (e != cudaSuccess) return e;
        k_fused_glob_rows_tc<__nv_bfloat16><<<grid, kTcThreads, smem, st>>>(mk, mv, a);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_global_proj(DType dt, const GlobalProjArgs &a, bool bwd, cudaStream_t st) {
    if (a.BH > 65535) return cudaErrorInvalidValue;   // grid z / y
    if (dt == kF32) return bwd ? launch_bwd_t<float>(a, st) : launch_fwd_t<float>(a, st);
    if (dt == kF16) return bwd ? launch_bwd_t<__half>(a, st) : launch_fwd_t<__half>(a, st);
    return bwd ? launch_bwd_t<__nv_bfloat16>(a, st) : launch_fwd_t<__nv_bfloat16>(a, st);
}

}  // namespace swab
