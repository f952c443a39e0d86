// k_global_proj.cu -- global queries with their own projections (ONNX Runtime
// issue "[WIP] Improve LongformerAttention performance", item (3): the
// global_q projection computed only for the G global tokens -- a compact Qg --
// with separate global key and value projections Kg, Vg over every position).
//
//   forward:  Og[g] = softmax_j(scale Qg[g].Kg[j]) Vg,  lseg[g]
//   backward: delta_g = dOg[g].Og[g];  ds_gj = p_gj (dOg[g].Vg[j] - delta_g)
//             dQg = scale ds Kg,  dKg = scale ds^T Qg,  dVg = p^T dOg
//
// G is a handful of tokens, so every product has G as one dimension and costs
// G * n * 64 multiply-adds per slice: FFMA with fp32 operands staged in shared
// memory (a 16-query chunk against 64-key tiles).  Parallelism comes from the
// keys: the forward splits them into chunks of kChunkKeys with per-chunk
// partial (max, sum, accumulator) merged by a second kernel; the backward
// gives each CTA one 64-key tile and every global query, so dKg, dVg rows have
// one writer, and its dQg partials are summed by a second kernel.  Both
// partial sets live in the caller's workspace.
#include "swab_internal.h"

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
__device__ __forceinline__ void load_rows(float *dst, const T *src, int row0, int nrows, int limit) {
    constexpr int V = 16 / sizeof(T);   // elements per 16-byte load
    for (int e = threadIdx.x; e < nrows * (64 / V); e += kThreads) {
        const int r = e / (64 / V), c0 = (e % (64 / V)) * V;
        const int row = row0 + r;
        float *d = dst + r * kPad + c0;
        if (row < limit) {
            const uint4 v = ldg16(reinterpret_cast<const uint4 *>(src + (long long)row * 64 + c0));
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
__device__ __forceinline__ void fetch_tile(TileRegs<T> &r, const T *src, int row0, int limit) {
    constexpr int V = 16 / sizeof(T), PR = 64 / V;   // elements per piece, pieces per row
#pragma unroll
    for (int k = 0; k < TileRegs<T>::kPer; ++k) {
        const int e = threadIdx.x + kThreads * k;
        const int row = row0 + e / PR;
        r.v[k] = row < limit ? ldg16(reinterpret_cast<const uint4 *>(src + (long long)row * 64 + (e % PR) * V))
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
    load_rows(qs, Qg, gc * kGC, kGC, G);
    const float xs = p.scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);   // channels 4 sub .. + 3
    const int k0 = kc * kChunkKeys, k1 = min(n, k0 + kChunkKeys);
    TileRegs<T> kr, vr;
    fetch_tile(kr, Kg, k0, n);
    fetch_tile(vr, Vg, k0, n);
    for (int j0 = k0; j0 < k1; j0 += kKT) {
        __syncthreads();   // the previous tile's readers are done
        store_tile(ks, kr);
        store_tile(vs, vr);
        if (j0 + kKT < k1) {   // the next tile's loads fly during this tile's products
            fetch_tile(kr, Kg, j0 + kKT, n);
            fetch_tile(vr, Vg, j0 + kKT, n);
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
        part[0] = m;
        part[1] = l;
    }
    part[2 + 4 * sub] = acc.x;
    part[3 + 4 * sub] = acc.y;
    part[4 + 4 * sub] = acc.z;
    part[5 + 4 * sub] = acc.w;
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
    for (int k = lane; k < p.nchunks; k += 32) M = fmaxf(M, base[k * step]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int k = lane; k < p.nchunks; k += 32) L = fmaf(base[k * step + 1], ex2(base[k * step] - M), L);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    float o0 = 0.f, o1 = 0.f;
    int k = 0;
    for (; k + 8 <= p.nchunks; k += 8) {
        float f[8], a[8], b[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float *c = base + (k + u) * step;
            f[u] = c[0];
            a[u] = c[2 + 2 * lane];
            b[u] = c[3 + 2 * lane];
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
        const float w = ex2(c[0] - M);
        o0 = fmaf(c[2 + 2 * lane], w, o0);
        o1 = fmaf(c[3 + 2 * lane], w, o1);
    }
    const float inv = 1.f / L;
    T *o = reinterpret_cast<T *>(p.Og) + bg * 64 + 2 * lane;
    o[0] = Elt<T>::from_f(o0 * inv);
    o[1] = Elt<T>::from_f(o1 * inv);
    if (lane == 0 && p.lseg) p.lseg[bg] = M / kLog2e + logf(L);
}

// ---------------------------------------------------------------------------
// backward: CTA (key tile, slice) over every global query
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
    load_rows(ks, Kg, j0, kKT, n);
    load_rows(vs, Vg, j0, kKT, n);
    // dK, dV of key jr = t / 4, channels 16 (t % 4) .. + 16
    const int jr = t >> 2, cq = (t & 3) * 16;
    float dk[16], dv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) dk[k] = dv[k] = 0.f;
    const float xs = p.scale * kLog2e;
    for (int g0 = 0; g0 < G; g0 += kGC) {
        __syncthreads();   // the previous chunk's readers are done
        load_rows(qs, Qg, g0, kGC, G);
        load_rows(dos, dOg, g0, kGC, G);
        if (t < kGC) lse_s[t] = g0 + t < G ? p.lseg[(long long)bh * G + g0 + t] * kLog2e : 0.f;
        // delta_g = dOg[g].Og[g]: 16 threads per query, 4 channels each
        {
            float d = 0.f;
            if (g0 + g < G) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = sub + 16 * u;
                    d = fmaf(Elt<T>::to_f(dOg[(long long)(g0 + g) * 64 + c]),
                             Elt<T>::to_f(Og[(long long)(g0 + g) * 64 + c]), d);
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
            *reinterpret_cast<float4 *>(part) =
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
        dK[k] = Elt<T>::from_f(p.scale * dk[k]);
        dV[k] = Elt<T>::from_f(dv[k]);
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
        for (int u = 0; u < 8; ++u) v[u] = base[(k + u) * step];
#pragma unroll
        for (int u = 0; u < 8; ++u) s += v[u];
    }
    for (; k < p.nchunks; ++k) s += base[k * step];
    reinterpret_cast<T *>(p.dQg)[e] = Elt<T>::from_f(s);
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
    const size_t fwd = (size_t)BH * ((n + kChunkKeys - 1) / kChunkKeys) * G * 66 * sizeof(float);
    const size_t bwd = (size_t)BH * ((n + kKT - 1) / kKT) * G * 64 * sizeof(float);
    return fwd > bwd ? fwd : bwd;
}

cudaError_t launch_global_proj(DType dt, const GlobalProjArgs &a, bool bwd, cudaStream_t st) {
    if (a.BH > 65535) return cudaErrorInvalidValue;   // grid z / y
    if (dt == kF32) return bwd ? launch_bwd_t<float>(a, st) : launch_fwd_t<float>(a, st);
    if (dt == kF16) return bwd ? launch_bwd_t<__half>(a, st) : launch_fwd_t<__half>(a, st);
    return bwd ? launch_bwd_t<__nv_bfloat16>(a, st) : launch_fwd_t<__nv_bfloat16>(a, st);
}

}  // namespace swab
