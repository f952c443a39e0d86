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
// Dropout (nvFuser issue, fusion 1: the kept probabilities scaled by
// 1/(1-p)): the forward also writes Pd = f * P, f the keep-and-scale factor of
// the slot's key, and the backward, given P and the gradient dP of Pd, forms
// dS = P * (f dP - delta_i), delta_i = sum P*f*dP.  A row's keep bits come
// from one Philox4x64-10 block per 32 keys of its residue (the lanes draw the
// blocks, one word of 32 bits each, into shared memory).
//
// One warp per band row.  A row of D elements starts at an arbitrary element
// boundary, so the warp walks the row's aligned 16-byte pieces (128-bit
// loads, 32 consecutive pieces per warp instruction).  All index math is
// 32-bit and relative to the row's first aligned piece; a piece whose
// elements are all valid takes a path with no per-element tests.  Pieces that
// straddle a row boundary are shared with the neighbouring row's warp: they
// are read whole but written element by element (only this row's elements);
// every other piece is written with one 128-bit store.
// Rows of at most 17 pieces per lane are read once into registers; longer
// rows stream twice (the second read hits L1/L2).
// exp is computed as 2^(x*log2(e) - m*log2(e)) with the ex2.approx
// instruction (relative error about 2^-22).
#include "swab_internal.h"

static constexpr unsigned kSwabFile = 6;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kRowsPerBlock = 4;  // warps per CTA
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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

// A band row in "piece coordinates": element x of the row's first aligned
// piece is slot x - lead.  Valid slots map to x in [xlo, xhi]; the row's own
// elements are x in [lead, lead + D).
struct Row {
    long long piece0;  // index (in 16-byte pieces) of the first piece touching the row
    int lead, npieces, xlo, xhi, xend;
};

template <typename T>
__device__ __forceinline__ Row make_row(const Geom &g, int R) {
    constexpr int N = Vec<T>::N;
    Row rw;
    const int i = R % g.n;
    const int t_lo = max(0, g.w - i / g.s);
    const int t_hi = min(g.D - 1, g.w + (g.n - 1 - i) / g.s);
    const long long e0 = (long long)R * g.D;
    rw.lead = (int)(e0 & (N - 1));
    rw.piece0 = e0 / N;
    rw.npieces = (rw.lead + g.D + N - 1) / N;
    rw.xlo = t_lo + rw.lead;
    rw.xhi = t_hi + rw.lead;
    rw.xend = rw.lead + g.D;
    return rw;
}

template <typename T>
__device__ __forceinline__ void store_piece(const Geom &g, uint4 *out, int pc, const Row &rw,
                                            const float (&y)[Vec<T>::N]) {
    constexpr int N = Vec<T>::N;
    const int x0 = pc * N;
    if (x0 >= rw.lead && x0 + N <= rw.xend) {
        *GP(g.bnd, out + pc) = pack<T>(y);
    } else {
        T *e = reinterpret_cast<T *>(out + pc);
#pragma unroll
        for (int u = 0; u < N; ++u)
            if (x0 + u >= rw.lead && x0 + u < rw.xend) *GP(g.bnd, e + u) = Elt<T>::from_f(y[u]);
    }
}

__device__ __forceinline__ bool all_valid(int x0, int n, const Row &rw) {
    return x0 >= rw.xlo && x0 + n - 1 <= rw.xhi;
}

// Key-padding bias row of row R's batch (null without a bias).
__device__ __forceinline__ const float *bias_row(const Geom &g, int R) {
    return g.kbias ? g.kbias + (size_t)(R / g.n / g.h) * g.n : nullptr;
}

// Adds the key bias to the valid elements of a piece: element x is slot
// t = x - lead, whose key is i + (t - w) * s.
template <int N>
__device__ __forceinline__ void add_key_bias(float (&x)[N], int x0, const Row &rw, const float *brow,
                                             int i, const Geom &g) {
#pragma unroll
    for (int u = 0; u < N; ++u) {
        const int xx = x0 + u;
        if (xx >= rw.xlo && xx <= rw.xhi) x[u] += __ldg(GP(g.bnd, brow + i + (xx - rw.lead - g.w) * g.s));
    }
}

// Dropout keep bits of one row: element x (piece coordinates) of the row has
// key sub-index b = x + a - w - lead (a = floor(i/s)); bit (b - 32 kb0) of the
// word table holds its keep decision.
struct Keep {
    const uint32_t *words;
    int off;   // x + off = b - 32 kb0
    float scale;
};

// Words per row the table needs: the valid keys span at most D, so at most
// (D - 1) / 32 + 2 blocks.
__host__ __device__ __forceinline__ int keep_words(int D) { return (D - 1) / 32 + 2; }

// Draws row R's keep bits into this warp's table (all lanes take part).
__device__ __forceinline__ Keep make_keep(const Geom &g, int R, const Row &rw, uint32_t *words,
                                          int lane) {
    const int i = R % g.n, bh = R / g.n, a = i / g.s;
    const int b_lo = a - g.w + (rw.xlo - rw.lead), b_hi = a - g.w + (rw.xhi - rw.lead);
    const int kb0 = b_lo >> 5, nkb = (b_hi >> 5) - kb0 + 1;
    for (int k = lane; k < nkb; k += 32) {
        unsigned long long wv[4];
        philox4x64_10((unsigned long long)(kb0 + k), (unsigned long long)i, (unsigned long long)bh,
                      0, g.seed, 0, wv);
        words[k] = keep_bits32(wv, g.drop_t);
    }
    __syncwarp();
    Keep kp;
    kp.words = words;
    kp.off = a - g.w - rw.lead - 32 * kb0;
    kp.scale = 256.f / (256.f - (float)g.drop_t);
    return kp;
}

// Keep-and-scale factor of valid element x.
__device__ __forceinline__ float keep_factor(const Keep &kp, int x) {
    const int b = x + kp.off;
    return ((kp.words[b >> 5] >> (b & 31)) & 1u) ? kp.scale : 0.f;
}

// dP -> f * dP on the valid elements of a piece (the gradient reaching P
// through the dropout).
template <int N>
__device__ __forceinline__ void apply_keep(float (&y)[N], int x0, const Row &rw, const Keep &kp) {
#pragma unroll
    for (int u = 0; u < N; ++u)
        if (x0 + u >= rw.xlo && x0 + u <= rw.xhi) y[u] *= keep_factor(kp, x0 + u);
}

// Stores f * y for a piece of probabilities (0 on invalid slots).
template <typename T>
__device__ __forceinline__ void store_dropped(const Geom &g, uint4 *out, int pc, const Row &rw, const Keep &kp,
                                              const float (&y)[Vec<T>::N]) {
    constexpr int N = Vec<T>::N;
    const int x0 = pc * N;
    float yd[N];
#pragma unroll
    for (int u = 0; u < N; ++u)
        yd[u] = (x0 + u >= rw.xlo && x0 + u <= rw.xhi) ? y[u] * keep_factor(kp, x0 + u) : 0.f;
    store_piece<T>(g, out, pc, rw, yd);
}

// ---------------------------------------------------------------------------
// register-resident rows: CTA (4 rows of one slice, slice) -- the grid gives
// the row's position directly, no division by n.  Invalid elements are
// replaced once, right after the unpack (-inf in the forward, 0 in the
// backward), so every later step is uniform packed fp32x2 arithmetic.
// ---------------------------------------------------------------------------
// Row geometry of position i of slice bh (s == 1 skips the divisions).
template <typename T>
__device__ __forceinline__ Row make_row_at(const Geom &g, long long R, int i) {
    constexpr int N = Vec<T>::N;
    Row rw;
    const int a = g.s == 1 ? i : i / g.s, b = g.s == 1 ? g.n - 1 - i : (g.n - 1 - i) / g.s;
    const int t_lo = max(0, g.w - a);
    const int t_hi = min(g.D - 1, g.w + b);
    const long long e0 = R * g.D;
    rw.lead = (int)(e0 & (N - 1));
    rw.piece0 = e0 / N;
    rw.npieces = (rw.lead + g.D + N - 1) / N;
    rw.xlo = t_lo + rw.lead;
    rw.xhi = t_hi + rw.lead;
    rw.xend = rw.lead + g.D;
    return rw;
}

// x[u] = fill where element x0 + u is outside the valid range
template <int N>
__device__ __forceinline__ void mask_piece(float (&x)[N], int x0, const Row &rw, float fill) {
    if (all_valid(x0, N, rw)) return;
#pragma unroll
    for (int u = 0; u < N; ++u)
        if (x0 + u < rw.xlo || x0 + u > rw.xhi) x[u] = fill;
}

template <typename T, int NCH, bool kDrop>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_softmax_reg(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    constexpr bool kKeep = NCH * N <= 32;  // keep the row's values in registers
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const int qi = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (qi >= g.n) return;
    const long long R = (long long)blockIdx.y * g.n + qi;
    const Row rw = make_row_at<T>(g, R, qi);
    const float *brow = g.kbias ? g.kbias + (size_t)(blockIdx.y / g.h) * g.n : nullptr;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    uint4 raw[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        raw[k] = pc < rw.npieces ? ldg16(GP(g.bnd, src + pc)) : make_uint4(0, 0, 0, 0);
    }
    // the keep bits are drawn while the row's loads are in flight
    extern __shared__ uint32_t keep_smem[];
    Keep kp{};
    if constexpr (kDrop)
        kp = make_keep(g, (int)R, rw, keep_smem + (threadIdx.x >> 5) * keep_words(g.D), lane);
    // scores (plus the key bias), invalid elements -inf
    auto scores = [&](int k, float (&x)[N]) {
        const int x0 = (lane + 32 * k) * N;
        unpack<T>(raw[k], x);
        if (brow) add_key_bias(x, x0, rw, brow, qi, g);
        mask_piece<N>(x, x0, rw, -INFINITY);
    };
    float xs[kKeep ? NCH * N : 1];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N];
        scores(k, x);
#pragma unroll
        for (int u = 0; u < N; u += 2) m = max3(m, x[u], x[u + 1]);
        if constexpr (kKeep) {
#pragma unroll
            for (int u = 0; u < N; ++u) xs[k * N + u] = x[u];
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float mb = m * kLog2e;
    const uint64_t l2 = f2(kLog2e, kLog2e), nb2 = f2(-mb, -mb);
    // e = 2^(x log2e - m log2e) of a piece (0 on invalid elements)
    auto expo = [&](float (&x)[N]) {
#pragma unroll
        for (int u = 0; u < N; u += 2) {
            float y0, y1;
            f2split(fma2(f2(x[u], x[u + 1]), l2, nb2), y0, y1);
            x[u] = ex2(y0);
            x[u + 1] = ex2(y1);
        }
    };
    uint64_t z2 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N];
        if constexpr (kKeep) {
#pragma unroll
            for (int u = 0; u < N; ++u) x[u] = xs[k * N + u];
        } else {
            scores(k, x);
        }
        expo(x);
#pragma unroll
        for (int u = 0; u < N; u += 2) z2 = add2(z2, f2(x[u], x[u + 1]));
        if constexpr (kKeep) {
#pragma unroll
            for (int u = 0; u < N; ++u) xs[k * N + u] = x[u];
        }
    }
    float z0, z1;
    f2split(z2, z0, z1);
    float z = z0 + z1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float inv = 1.f / z;
    const uint64_t inv2 = f2(inv, inv);
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
    uint4 *dstd = reinterpret_cast<uint4 *>(p.Pd) + rw.piece0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        if (pc >= rw.npieces) break;
        float y[N];
        if constexpr (kKeep) {
#pragma unroll
            for (int u = 0; u < N; ++u) y[u] = xs[k * N + u];
        } else {
            scores(k, y);
            expo(y);
        }
#pragma unroll
        for (int u = 0; u < N; u += 2) f2split(mul2(f2(y[u], y[u + 1]), inv2), y[u], y[u + 1]);
        if constexpr (kDrop) {
            if (p.P) store_piece<T>(g, dst, pc, rw, y);
            store_dropped<T>(g, dstd, pc, rw, kp, y);
        } else {
            store_piece<T>(g, dst, pc, rw, y);
        }
    }
    if (p.lse && lane == 0) *GP(g.bnd, p.lse + R) = m + logf(z);
}

template <typename T, int NCH, bool kDrop>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_softmax_bwd_reg(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const int qi = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (qi >= g.n) return;
    const long long R = (long long)blockIdx.y * g.n + qi;
    const Row rw = make_row_at<T>(g, R, qi);
    const uint4 *sp = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    const uint4 *sd = reinterpret_cast<const uint4 *>(p.S2) + rw.piece0;
    uint4 rp[NCH], rd[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        const bool in = pc < rw.npieces;
        rp[k] = in ? ldg16(GP(g.bnd, sp + pc)) : make_uint4(0, 0, 0, 0);
        rd[k] = in ? ldg16(GP(g.bnd, sd + pc)) : make_uint4(0, 0, 0, 0);
    }
    // the keep bits are drawn while the row's loads are in flight
    extern __shared__ uint32_t keep_smem[];
    Keep kp{};
    if constexpr (kDrop)
        kp = make_keep(g, (int)R, rw, keep_smem + (threadIdx.x >> 5) * keep_words(g.D), lane);
    // P and the gradient reaching P (f dP with dropout) of a piece, both 0 on
    // invalid elements (whatever those slots hold)
    auto operands = [&](int k, float (&x)[N], float (&y)[N]) {
        const int x0 = (lane + 32 * k) * N;
        unpack<T>(rp[k], x);
        unpack<T>(rd[k], y);
        if constexpr (kDrop) apply_keep<N>(y, x0, rw, kp);
        mask_piece<N>(x, x0, rw, 0.f);
        mask_piece<N>(y, x0, rw, 0.f);
    };
    uint64_t d2 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N], y[N];
        operands(k, x, y);
#pragma unroll
        for (int u = 0; u < N; u += 2) d2 = fma2(f2(x[u], x[u + 1]), f2(y[u], y[u + 1]), d2);
    }
    float d0, d1;
    f2split(d2, d0, d1);
    float delta = d0 + d1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
    const uint64_t nd2 = f2(-delta, -delta);
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        if (pc >= rw.npieces) break;
        float x[N], y[N];
        operands(k, x, y);
#pragma unroll
        for (int u = 0; u < N; u += 2)
            f2split(mul2(f2(x[u], x[u + 1]), add2(f2(y[u], y[u + 1]), nd2)), x[u], x[u + 1]);
        store_piece<T>(g, dst, pc, rw, x);
    }
}

// ---------------------------------------------------------------------------
// long rows: one CTA of kWideThreads per row (grid (position, slice)), each
// thread holding at most NCH pieces -- the row is read once, one exp per
// element, and the max and sum reductions go across the CTA's warps
// through shared memory.  A warp per row would hold up to 17 pieces a lane
// and recompute the exponentials; spread over eight warps the row stays in
// registers.
// ---------------------------------------------------------------------------
constexpr int kWideThreads = 256;
constexpr int kWideWarps = kWideThreads / 32;

// max (kMax) or sum over the CTA; `red` holds kWideWarps floats
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = kMax ? fmaxf(v, o) : v + o;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kWideWarps; ++w) r = kMax ? fmaxf(r, red[w]) : r + red[w];
    __syncthreads();   // `red` is reused by the next reduction
    return r;
}

// The row's keep bits drawn by the whole CTA (the warp version's table).
__device__ __forceinline__ Keep make_keep_block(const Geom &g, int R, const Row &rw, uint32_t *words) {
    const int i = R % g.n, bh = R / g.n, a = i / g.s;
    const int b_lo = a - g.w + (rw.xlo - rw.lead), b_hi = a - g.w + (rw.xhi - rw.lead);
    const int kb0 = b_lo >> 5, nkb = (b_hi >> 5) - kb0 + 1;
    for (int k = threadIdx.x; k < nkb; k += blockDim.x) {
        unsigned long long wv[4];
        philox4x64_10((unsigned long long)(kb0 + k), (unsigned long long)i, (unsigned long long)bh,
                      0, g.seed, 0, wv);
        words[k] = keep_bits32(wv, g.drop_t);
    }
    __syncthreads();
    Keep kp;
    kp.words = words;
    kp.off = a - g.w - rw.lead - 32 * kb0;
    kp.scale = 256.f / (256.f - (float)g.drop_t);
    return kp;
}

template <typename T, int NCH, bool kDrop>
__global__ void __launch_bounds__(kWideThreads) k_softmax_wide(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    static_assert(NCH * N <= 32, "the row's values stay in registers");
    const Geom &g = p.g;
    const int tid = threadIdx.x;
    const int qi = blockIdx.x;
    const long long R = (long long)blockIdx.y * g.n + qi;
    const Row rw = make_row_at<T>(g, R, qi);
    const float *brow = g.kbias ? g.kbias + (size_t)(blockIdx.y / g.h) * g.n : nullptr;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    uint4 raw[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = tid + kWideThreads * k;
        raw[k] = pc < rw.npieces ? ldg16(GP(g.bnd, src + pc)) : make_uint4(0, 0, 0, 0);
    }
    __shared__ float red[kWideWarps];
    extern __shared__ uint32_t keep_smem[];
    Keep kp{};
    if constexpr (kDrop) kp = make_keep_block(g, (int)R, rw, keep_smem);
    // scores (plus the key bias), invalid elements -inf
    float xs[NCH * N];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N];
        const int x0 = (tid + kWideThreads * k) * N;
        unpack<T>(raw[k], x);
        if (brow) add_key_bias(x, x0, rw, brow, qi, g);
        mask_piece<N>(x, x0, rw, -INFINITY);
#pragma unroll
        for (int u = 0; u < N; u += 2) m = max3(m, x[u], x[u + 1]);
#pragma unroll
        for (int u = 0; u < N; ++u) xs[k * N + u] = x[u];
    }
    m = block_reduce<true>(m, red);
    const float mb = m * kLog2e;
    const uint64_t l2 = f2(kLog2e, kLog2e), nb2 = f2(-mb, -mb);
    uint64_t z2 = f2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < NCH * N; u += 2) {
        float y0, y1;
        f2split(fma2(f2(xs[u], xs[u + 1]), l2, nb2), y0, y1);
        xs[u] = ex2(y0);
        xs[u + 1] = ex2(y1);
        z2 = add2(z2, f2(xs[u], xs[u + 1]));
    }
    float z0, z1;
    f2split(z2, z0, z1);
    const float z = block_reduce<false>(z0 + z1, red);
    const float inv = 1.f / z;
    const uint64_t inv2 = f2(inv, inv);
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
    uint4 *dstd = reinterpret_cast<uint4 *>(p.Pd) + rw.piece0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = tid + kWideThreads * k;
        if (pc >= rw.npieces) break;
        float y[N];
#pragma unroll
        for (int u = 0; u < N; u += 2) f2split(mul2(f2(xs[k * N + u], xs[k * N + u + 1]), inv2), y[u], y[u + 1]);
        if constexpr (kDrop) {
            if (p.P) store_piece<T>(g, dst, pc, rw, y);
            store_dropped<T>(g, dstd, pc, rw, kp, y);
        } else {
            store_piece<T>(g, dst, pc, rw, y);
        }
    }
    if (p.lse && tid == 0) *GP(g.bnd, p.lse + R) = m + logf(z);
}

template <typename T, int NCH, bool kDrop>
__global__ void __launch_bounds__(kWideThreads) k_softmax_bwd_wide(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    static_assert(NCH * N <= 32, "the row's values stay in registers");
    const Geom &g = p.g;
    const int tid = threadIdx.x;
    const int qi = blockIdx.x;
    const long long R = (long long)blockIdx.y * g.n + qi;
    const Row rw = make_row_at<T>(g, R, qi);
    const uint4 *sp = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    const uint4 *sd = reinterpret_cast<const uint4 *>(p.S2) + rw.piece0;
    uint4 rp[NCH], rd[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = tid + kWideThreads * k;
        const bool in = pc < rw.npieces;
        rp[k] = in ? ldg16(GP(g.bnd, sp + pc)) : make_uint4(0, 0, 0, 0);
        rd[k] = in ? ldg16(GP(g.bnd, sd + pc)) : make_uint4(0, 0, 0, 0);
    }
    __shared__ float red[kWideWarps];
    extern __shared__ uint32_t keep_smem[];
    Keep kp{};
    if constexpr (kDrop) kp = make_keep_block(g, (int)R, rw, keep_smem);
    // P and the gradient reaching P (f dP with dropout), 0 on invalid elements
    float xp[NCH * N], yd[NCH * N];
    uint64_t d2 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N], y[N];
        const int x0 = (tid + kWideThreads * k) * N;
        unpack<T>(rp[k], x);
        unpack<T>(rd[k], y);
        if constexpr (kDrop) apply_keep<N>(y, x0, rw, kp);
        mask_piece<N>(x, x0, rw, 0.f);
        mask_piece<N>(y, x0, rw, 0.f);
#pragma unroll
        for (int u = 0; u < N; u += 2) d2 = fma2(f2(x[u], x[u + 1]), f2(y[u], y[u + 1]), d2);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            xp[k * N + u] = x[u];
            yd[k * N + u] = y[u];
        }
    }
    float d0, d1;
    f2split(d2, d0, d1);
    const float delta = block_reduce<false>(d0 + d1, red);
    const uint64_t nd2 = f2(-delta, -delta);
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = tid + kWideThreads * k;
        if (pc >= rw.npieces) break;
        float x[N];
#pragma unroll
        for (int u = 0; u < N; u += 2)
            f2split(mul2(f2(xp[k * N + u], xp[k * N + u + 1]), add2(f2(yd[k * N + u], yd[k * N + u + 1]), nd2)),
                    x[u], x[u + 1]);
        store_piece<T>(g, dst, pc, rw, x);
    }
}

// ---------------------------------------------------------------------------
// streaming rows (longer than the register path holds): two reads
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_softmax_stream(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const int R = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (R >= g.BH * g.n) return;
    const Row rw = make_row<T>(g, R);
    const float *brow = bias_row(g, R);
    const int qi = R % g.n;
    const bool drop = p.Pd != nullptr;
    extern __shared__ uint32_t keep_smem[];
    Keep kp{};
    if (drop) kp = make_keep(g, R, rw, keep_smem + (threadIdx.x >> 5) * keep_words(g.D), lane);
    const uint4 *src = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    // pass 1: per-lane running max (log2 units) and sum, one rescale per piece
    float m = -INFINITY, z = 0.f;
    for (int pc = lane; pc < rw.npieces; pc += 32) {
        float x[N];
        unpack<T>(ldg16(GP(g.bnd, src + pc)), x);
        const int x0 = pc * N;
        if (brow) add_key_bias(x, x0, rw, brow, qi, g);
        float pm = -INFINITY;
#pragma unroll
        for (int u = 0; u < N; ++u) {
            x[u] *= kLog2e;
            if (x0 + u >= rw.xlo && x0 + u <= rw.xhi) pm = fmaxf(pm, x[u]);
        }
        if (pm == -INFINITY) continue;
        const float mn = fmaxf(m, pm);
        z = (m == -INFINITY) ? 0.f : z * ex2(m - mn);
#pragma unroll
        for (int u = 0; u < N; ++u)
            if (x0 + u >= rw.xlo && x0 + u <= rw.xhi) z += ex2(x[u] - mn);
        m = mn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
        const float mn = fmaxf(m, m2);
        z = (m == -INFINITY ? 0.f : z * ex2(m - mn)) + (m2 == -INFINITY ? 0.f : z2 * ex2(m2 - mn));
        m = mn;
    }
    const float inv = 1.f / z;
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
    uint4 *dstd = reinterpret_cast<uint4 *>(p.Pd) + rw.piece0;
    for (int pc = lane; pc < rw.npieces; pc += 32) {
        float x[N];
        unpack<T>(ldg16(GP(g.bnd, src + pc)), x);
        const int x0 = pc * N;
        if (brow) add_key_bias(x, x0, rw, brow, qi, g);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const bool v = x0 + u >= rw.xlo && x0 + u <= rw.xhi;
            x[u] = v ? ex2(fmaf(x[u], kLog2e, -m)) * inv : 0.f;
        }
        if (p.P) store_piece<T>(g, dst, pc, rw, x);
        if (drop) store_dropped<T>(g, dstd, pc, rw, kp, x);
    }
    if (p.lse && lane == 0) *GP(g.bnd, p.lse + R) = m / kLog2e + logf(z);
}

template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_softmax_bwd_stream(const SoftmaxArgs p) {
    constexpr int N = Vec<T>::N;
    const Geom &g = p.g;
    const int lane = threadIdx.x & 31;
    const int R = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (R >= g.BH * g.n) return;
    const Row rw = make_row<T>(g, R);
    const bool drop = g.drop_t > 0;
    extern __shared__ uint32_t keep_smem[];
    Keep kp{};
    if (drop) kp = make_keep(g, R, rw, keep_smem + (threadIdx.x >> 5) * keep_words(g.D), lane);
    const uint4 *sp = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    const uint4 *sd = reinterpret_cast<const uint4 *>(p.S2) + rw.piece0;
    float delta = 0.f;
    for (int pc = lane; pc < rw.npieces; pc += 32) {
        float x[N], y[N];
        unpack<T>(ldg16(GP(g.bnd, sp + pc)), x);
        unpack<T>(ldg16(GP(g.bnd, sd + pc)), y);
        const int x0 = pc * N;
        if (drop) apply_keep<N>(y, x0, rw, kp);
#pragma unroll
        for (int u = 0; u < N; ++u)
            if (x0 + u >= rw.xlo && x0 + u <= rw.xhi) delta = fmaf(x[u], y[u], delta);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
    for (int pc = lane; pc < rw.npieces; pc += 32) {
        float x[N], y[N];
        unpack<T>(ldg16(GP(g.bnd, sp + pc)), x);
        unpack<T>(ldg16(GP(g.bnd, sd + pc)), y);
        const int x0 = pc * N;
        if (drop) apply_keep<N>(y, x0, rw, kp);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const bool v = x0 + u >= rw.xlo && x0 + u <= rw.xhi;
            x[u] = v ? x[u] * (y[u] - delta) : 0.f;
        }
        store_piece<T>(g, dst, pc, rw, x);
    }
}

// ---------------------------------------------------------------------------
// Softmax with global tokens ("[WIP] Improve LongformerAttention performance",
// ONNX Runtime issue, item (1)).  A local row i takes its band slots whose key
// is in the sequence and not global, plus its G values at the global keys
// (the cols piece [BH, n, G]); a global row's band and cols rows are zero (its
// softmax is the dense row, [BH, G, n], done apart).  Warp per band row,
// 16-byte pieces in registers as in the plain kernels; a piece tests its keys
// against the global index only when its key span reaches the index's range.
// ---------------------------------------------------------------------------
constexpr int kColsPerLane = (kMaxGlobal + 31) / 32;

template <typename T> __device__ __forceinline__ float ld(const T *p) { return Elt<T>::to_f(*p); }

__device__ __forceinline__ bool is_global_pos(const GlobArgs &gl, long long j) {
    if (j < gl.idx[0] || j > gl.idx[gl.G - 1]) return false;
    int lo = 0, hi = gl.G - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (gl.idx[mid] < j) lo = mid + 1;
        else hi = mid;
    }
    return gl.idx[lo] == j;
}

// x[u] = fill where element x0 + u's key (i + (x - lead - w) s) is global
template <int N>
__device__ __forceinline__ void mask_global_keys(float (&x)[N], int x0, const Row &rw, int i, const Geom &g,
                                                 const GlobArgs &gl, float fill) {
    const long long j0 = (long long)i + (long long)(x0 - rw.lead - g.w) * g.s;
    const long long j1 = j0 + (long long)(N - 1) * g.s;
    if (j1 < gl.idx[0] || j0 > gl.idx[gl.G - 1]) return;
#pragma unroll
    for (int u = 0; u < N; ++u)
        if (is_global_pos(gl, j0 + (long long)u * g.s)) x[u] = fill;
}

template <typename T, int NCH>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_softmax_glob_reg(const SoftmaxGlobArgs p) {
    constexpr int N = Vec<T>::N;
    static_assert(NCH * N <= 32, "the row's values stay in registers");
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int lane = threadIdx.x & 31;
    const int qi = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (qi >= g.n) return;
    const long long R = (long long)blockIdx.y * g.n + qi;
    const Row rw = make_row_at<T>(g, R, qi);
    const int G = gl.G;
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
    T *pcol = reinterpret_cast<T *>(p.Pcols) + R * G;
    if (is_global_pos(gl, qi)) {
        float zero[N];
#pragma unroll
        for (int u = 0; u < N; ++u) zero[u] = 0.f;
        for (int pc = lane; pc < rw.npieces; pc += 32) store_piece<T>(g, dst, pc, rw, zero);
        for (int q = lane; q < G; q += 32) *GP(g.bnd, pcol + q) = Elt<T>::from_f(0.f);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    uint4 raw[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        raw[k] = pc < rw.npieces ? ldg16(GP(g.bnd, src + pc)) : make_uint4(0, 0, 0, 0);
    }
    const T *scol = reinterpret_cast<const T *>(p.Scols) + R * G;
    float cv[kColsPerLane];
#pragma unroll
    // the key bias (band slots and the global columns' keys G[q])
    const float *brow = g.kbias ? g.kbias + (size_t)(blockIdx.y / g.h) * g.n : nullptr;
    for (int k = 0; k < kColsPerLane; ++k) {
        const int q = lane + 32 * k;
        cv[k] = q < G ? ld(GP(g.bnd, scol + q)) + (brow ? __ldg(GP(g.bnd, brow + gl.idx[q])) : 0.f) : -INFINITY;
    }
    float xs[NCH * N];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N];
        const int x0 = (lane + 32 * k) * N;
        unpack<T>(raw[k], x);
        if (brow) add_key_bias(x, x0, rw, brow, qi, g);
        mask_piece<N>(x, x0, rw, -INFINITY);
        mask_global_keys<N>(x, x0, rw, qi, g, gl, -INFINITY);
#pragma unroll
        for (int u = 0; u < N; u += 2) m = max3(m, x[u], x[u + 1]);
#pragma unroll
        for (int u = 0; u < N; ++u) xs[k * N + u] = x[u];
    }
#pragma unroll
    for (int k = 0; k < kColsPerLane; ++k) m = fmaxf(m, cv[k]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float mb = m * kLog2e;
    const uint64_t l2 = f2(kLog2e, kLog2e), nb2 = f2(-mb, -mb);
    uint64_t z2 = f2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < NCH * N; u += 2) {
        float y0, y1;
        f2split(fma2(f2(xs[u], xs[u + 1]), l2, nb2), y0, y1);
        xs[u] = ex2(y0);
        xs[u + 1] = ex2(y1);
        z2 = add2(z2, f2(xs[u], xs[u + 1]));
    }
    float z0, z1;
    f2split(z2, z0, z1);
    float z = z0 + z1;
#pragma unroll
    for (int k = 0; k < kColsPerLane; ++k) {
        cv[k] = ex2(fmaf(cv[k], kLog2e, -mb));
        z += cv[k];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float inv = 1.f / z;
    const uint64_t inv2 = f2(inv, inv);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        if (pc >= rw.npieces) break;
        float y[N];
#pragma unroll
        for (int u = 0; u < N; u += 2) f2split(mul2(f2(xs[k * N + u], xs[k * N + u + 1]), inv2), y[u], y[u + 1]);
        store_piece<T>(g, dst, pc, rw, y);
    }
#pragma unroll
    for (int k = 0; k < kColsPerLane; ++k) {
        const int q = lane + 32 * k;
        if (q < G) *GP(g.bnd, pcol + q) = Elt<T>::from_f(cv[k] * inv);
    }
    if (p.lse && lane == 0) *GP(g.bnd, p.lse + R) = m + logf(z);
}

// dS = P (dP - delta) on the used slots and dSc = Pc (dPc - delta) on the
// cols, delta = sum over both of P dP; a global row's band and cols rows are 0
template <typename T, int NCH>
__global__ void __launch_bounds__(kRowsPerBlock * 32) k_softmax_bwd_glob_reg(const SoftmaxGlobArgs p) {
    constexpr int N = Vec<T>::N;
    static_assert(NCH * N <= 32, "the row's values stay in registers");
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int lane = threadIdx.x & 31;
    const int qi = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (qi >= g.n) return;
    const long long R = (long long)blockIdx.y * g.n + qi;
    const Row rw = make_row_at<T>(g, R, qi);
    const int G = gl.G;
    uint4 *dst = reinterpret_cast<uint4 *>(p.P) + rw.piece0;
    T *dscol = reinterpret_cast<T *>(p.Pcols) + R * G;
    if (is_global_pos(gl, qi)) {
        float zero[N];
#pragma unroll
        for (int u = 0; u < N; ++u) zero[u] = 0.f;
        for (int pc = lane; pc < rw.npieces; pc += 32) store_piece<T>(g, dst, pc, rw, zero);
        for (int q = lane; q < G; q += 32) *GP(g.bnd, dscol + q) = Elt<T>::from_f(0.f);
        return;
    }
    const uint4 *sp = reinterpret_cast<const uint4 *>(p.S) + rw.piece0;
    const uint4 *sd = reinterpret_cast<const uint4 *>(p.S2) + rw.piece0;
    uint4 rp[NCH], rd[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        const bool in = pc < rw.npieces;
        rp[k] = in ? ldg16(GP(g.bnd, sp + pc)) : make_uint4(0, 0, 0, 0);
        rd[k] = in ? ldg16(GP(g.bnd, sd + pc)) : make_uint4(0, 0, 0, 0);
    }
    const T *pcol = reinterpret_cast<const T *>(p.Scols) + R * G;
    const T *dpcol = reinterpret_cast<const T *>(p.S2cols) + R * G;
    float pv[kColsPerLane], dv[kColsPerLane];
#pragma unroll
    for (int k = 0; k < kColsPerLane; ++k) {
        const int q = lane + 32 * k;
        pv[k] = q < G ? ld(GP(g.bnd, pcol + q)) : 0.f;
        dv[k] = q < G ? ld(GP(g.bnd, dpcol + q)) : 0.f;
    }
    float xp[NCH * N], yd[NCH * N];
    uint64_t d2 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        float x[N], y[N];
        const int x0 = (lane + 32 * k) * N;
        unpack<T>(rp[k], x);
        unpack<T>(rd[k], y);
        mask_piece<N>(x, x0, rw, 0.f);
        mask_piece<N>(y, x0, rw, 0.f);
        mask_global_keys<N>(x, x0, rw, qi, g, gl, 0.f);
        mask_global_keys<N>(y, x0, rw, qi, g, gl, 0.f);
#pragma unroll
        for (int u = 0; u < N; u += 2) d2 = fma2(f2(x[u], x[u + 1]), f2(y[u], y[u + 1]), d2);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            xp[k * N + u] = x[u];
            yd[k * N + u] = y[u];
        }
    }
    float d0, d1;
    f2split(d2, d0, d1);
    float delta = d0 + d1;
#pragma unroll
    for (int k = 0; k < kColsPerLane; ++k) delta = fmaf(pv[k], dv[k], delta);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) delta += __shfl_xor_sync(0xffffffffu, delta, off);
    const uint64_t nd2 = f2(-delta, -delta);
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int pc = lane + 32 * k;
        if (pc >= rw.npieces) break;
        float x[N];
#pragma unroll
        for (int u = 0; u < N; u += 2)
            f2split(mul2(f2(xp[k * N + u], xp[k * N + u + 1]), add2(f2(yd[k * N + u], yd[k * N + u + 1]), nd2)),
                    x[u], x[u + 1]);
        store_piece<T>(g, dst, pc, rw, x);
    }
#pragma unroll
    for (int k = 0; k < kColsPerLane; ++k) {
        const int q = lane + 32 * k;
        if (q < G) *GP(g.bnd, dscol + q) = Elt<T>::from_f(pv[k] * (dv[k] - delta));
    }
}

// Dense softmax (and its backward) of the G global query rows [BH, G, n]: a
// CTA of kWideThreads per row, 16-byte pieces (n a multiple of a piece), at
// most NCH pieces a thread.
template <typename T, int NCH, bool kBwd>
__global__ void __launch_bounds__(kWideThreads) k_glob_rows_wide(const SoftmaxGlobArgs p) {
    constexpr int N = Vec<T>::N;
    static_assert(NCH * N <= 32, "the row's values stay in registers");
    const Geom &g = p.g;
    const GlobArgs &gl = p.gl;
    const int tid = threadIdx.x;
    const long long W = blockIdx.x;   // (slice, g)
    const int np = g.n / N;
    __shared__ float red[kWideWarps];
    const uint4 *x4 = reinterpret_cast<const uint4 *>(p.Srows) + W * np;
    uint4 *y4 = reinterpret_cast<uint4 *>(p.Prows) + W * np;
    float xs[NCH * N];
    if constexpr (!kBwd) {
        // plus the key bias of every key (the row spans the sequence)
        const float *brow = g.kbias ? g.kbias + (size_t)(W / gl.G / g.h) * g.n : nullptr;
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int pc = tid + kWideThreads * k;
            float x[N];
            unpack<T>(pc < np ? ldg16(GP(g.bnd, x4 + pc)) : make_uint4(0, 0, 0, 0), x);
            if (brow && pc < np) {
#pragma unroll
                for (int u = 0; u < N; ++u) x[u] += __ldg(GP(g.bnd, brow + (size_t)pc * N + u));
            }
#pragma unroll
            for (int u = 0; u < N; ++u) {
                xs[k * N + u] = pc < np ? x[u] : -INFINITY;
                m = fmaxf(m, xs[k * N + u]);
            }
        }
        m = block_reduce<true>(m, red);
        const float mb = m * kLog2e;
        float z = 0.f;
#pragma unroll
        for (int u = 0; u < NCH * N; ++u) {
            xs[u] = ex2(fmaf(xs[u], kLog2e, -mb));
            z += xs[u];
        }
        z = block_reduce<false>(z, red);
        const float inv = 1.f / z;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int pc = tid + kWideThreads * k;
            if (pc >= np) break;
            float y[N];
#pragma unroll
            for (int u = 0; u < N; ++u) y[u] = xs[k * N + u] * inv;
            *GP(g.bnd, y4 + pc) = pack<T>(y);
        }
        if (p.lse && tid == 0) *GP(g.bnd, p.lse + (W / gl.G) * g.n + gl.idx[W % gl.G]) = m + logf(z);
    } else {
        const uint4 *d4 = reinterpret_cast<const uint4 *>(p.S2rows) + W * np;
        float ys[NCH * N];
        float delta = 0.f;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int pc = tid + kWideThreads * k;
            float x[N], y[N];
            unpack<T>(pc < np ? ldg16(GP(g.bnd, x4 + pc)) : make_uint4(0, 0, 0, 0), x);
            unpack<T>(pc < np ? ldg16(GP(g.bnd, d4 + pc)) : make_uint4(0, 0, 0, 0), y);
#pragma unroll
            for (int u = 0; u < N; ++u) {
                xs[k * N + u] = x[u];
                ys[k * N + u] = y[u];
                delta = fmaf(x[u], y[u], delta);
            }
        }
        delta = block_reduce<false>(delta, red);
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int pc = tid + kWideThreads * k;
            if (pc >= np) break;
            float y[N];
#pragma unroll
            for (int u = 0; u < N; ++u) y[u] = xs[k * N + u] * (ys[k * N + u] - delta);
            *GP(g.bnd, y4 + pc) = pack<T>(y);
        }
    }
}

template <typename T>
bool launch_glob_fast_t(const SoftmaxGlobArgs &a, bool bwd, cudaStream_t st, cudaError_t *err,
                        bool *rows_done) {
    constexpr int N = Vec<T>::N;
    const long long pieces = (a.g.D + N - 1) / N + 1;
    const long long per_lane = (pieces + 31) / 32;
    if (per_lane * N > 32 || a.gl.G < 1) return false;
    const int rp = a.g.n / N;
    const bool rows_fast = a.g.n % N == 0 && (rp + kWideThreads - 1) / kWideThreads * N <= 32;
    const dim3 grd2((unsigned)((a.g.n + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)a.g.BH);
    const dim3 blk(kRowsPerBlock * 32);
    constexpr int kMaxNch = 32 / N;
    if (bwd) {
        if (per_lane <= 1) k_softmax_bwd_glob_reg<T, 1><<<grd2, blk, 0, st>>>(a);
        else if (per_lane <= 2) k_softmax_bwd_glob_reg<T, 2><<<grd2, blk, 0, st>>>(a);
        else k_softmax_bwd_glob_reg<T, kMaxNch><<<grd2, blk, 0, st>>>(a);
    } else {
        if (per_lane <= 1) k_softmax_glob_reg<T, 1><<<grd2, blk, 0, st>>>(a);
        else if (per_lane <= 2) k_softmax_glob_reg<T, 2><<<grd2, blk, 0, st>>>(a);
        else k_softmax_glob_reg<T, kMaxNch><<<grd2, blk, 0, st>>>(a);
    }
    *err = cudaGetLastError();
    *rows_done = rows_fast;
    if (*err != cudaSuccess || !rows_fast) return true;   // the dense rows: done by the caller
    const unsigned rows = (unsigned)((long long)a.g.BH * a.gl.G);
    const int per_thread = (rp + kWideThreads - 1) / kWideThreads;
    if (bwd) {
        if (per_thread <= 1) k_glob_rows_wide<T, 1, true><<<rows, kWideThreads, 0, st>>>(a);
        else if (per_thread <= 2) k_glob_rows_wide<T, 2, true><<<rows, kWideThreads, 0, st>>>(a);
        else k_glob_rows_wide<T, kMaxNch, true><<<rows, kWideThreads, 0, st>>>(a);
    } else {
        if (per_thread <= 1) k_glob_rows_wide<T, 1, false><<<rows, kWideThreads, 0, st>>>(a);
        else if (per_thread <= 2) k_glob_rows_wide<T, 2, false><<<rows, kWideThreads, 0, st>>>(a);
        else k_glob_rows_wide<T, kMaxNch, false><<<rows, kWideThreads, 0, st>>>(a);
    }
    *err = cudaGetLastError();
    return true;
}

template <typename T, bool kDrop>
cudaError_t launch_sm_v(const SoftmaxArgs &a, bool bwd, cudaStream_t st) {
    constexpr int N = Vec<T>::N;
    const long long rows = (long long)a.g.BH * a.g.n;
    const dim3 grd((unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock));   // streaming kernels
    const dim3 grd2((unsigned)((a.g.n + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)a.g.BH);
    const dim3 blk(kRowsPerBlock * 32);
    const long long pieces = (a.g.D + N - 1) / N + 1;  // most pieces a row touches
    const long long per_lane = (pieces + 31) / 32;
    // dropout: each warp's keep-bit table for its row
    const size_t smem = kDrop ? (size_t)kRowsPerBlock * keep_words(a.g.D) * sizeof(uint32_t) : 0;
    // rows past four pieces a lane: a CTA per row while its pieces fit the
    // CTA's registers (at most 32 values a thread)
    const long long per_thread = (pieces + kWideThreads - 1) / kWideThreads;
    if (per_lane > 4 && per_thread * N <= 32) {
        const dim3 grw((unsigned)a.g.n, (unsigned)a.g.BH);
        const size_t smw = kDrop ? (size_t)keep_words(a.g.D) * sizeof(uint32_t) : 0;
        if (bwd) {
            if (per_thread <= 1) k_softmax_bwd_wide<T, 1, kDrop><<<grw, kWideThreads, smw, st>>>(a);
            else if (per_thread <= 2) k_softmax_bwd_wide<T, 2, kDrop><<<grw, kWideThreads, smw, st>>>(a);
            else if (per_thread <= 4) k_softmax_bwd_wide<T, 4, kDrop><<<grw, kWideThreads, smw, st>>>(a);
            else k_softmax_bwd_wide<T, 32 / N, kDrop><<<grw, kWideThreads, smw, st>>>(a);
        } else {
            if (per_thread <= 1) k_softmax_wide<T, 1, kDrop><<<grw, kWideThreads, smw, st>>>(a);
            else if (per_thread <= 2) k_softmax_wide<T, 2, kDrop><<<grw, kWideThreads, smw, st>>>(a);
            else if (per_thread <= 4) k_softmax_wide<T, 4, kDrop><<<grw, kWideThreads, smw, st>>>(a);
            else k_softmax_wide<T, 32 / N, kDrop><<<grw, kWideThreads, smw, st>>>(a);
        }
        return cudaGetLastError();
    }
    if (bwd) {
        if (per_lane <= 1) k_softmax_bwd_reg<T, 1, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 2) k_softmax_bwd_reg<T, 2, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 3) k_softmax_bwd_reg<T, 3, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 4) k_softmax_bwd_reg<T, 4, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 8) k_softmax_bwd_reg<T, 8, kDrop><<<grd2, blk, smem, st>>>(a);
        else k_softmax_bwd_stream<T><<<grd, blk, smem, st>>>(a);
    } else {
        if (per_lane <= 1) k_softmax_reg<T, 1, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 2) k_softmax_reg<T, 2, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 3) k_softmax_reg<T, 3, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 4) k_softmax_reg<T, 4, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 8) k_softmax_reg<T, 8, kDrop><<<grd2, blk, smem, st>>>(a);
        else if (per_lane <= 17) k_softmax_reg<T, 17, kDrop><<<grd2, blk, smem, st>>>(a);
        else k_softmax_stream<T><<<grd, blk, smem, st>>>(a);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_sm(const SoftmaxArgs &a, bool bwd, cudaStream_t st) {
    const bool drop = bwd ? a.g.drop_t > 0 : a.Pd != nullptr;
    return drop ? launch_sm_v<T, true>(a, bwd, st) : launch_sm_v<T, false>(a, bwd, st);
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

bool launch_softmax_glob_fast(DType dt, const SoftmaxGlobArgs &a, bool bwd, bool *rows_done,
                              cudaStream_t st, cudaError_t *err) {
    *rows_done = false;
    if (dt == kF32) return launch_glob_fast_t<float>(a, bwd, st, err, rows_done);
    if (dt == kF16) return launch_glob_fast_t<__half>(a, bwd, st, err, rows_done);
    return launch_glob_fast_t<__nv_bfloat16>(a, bwd, st, err, rows_done);
}

}  // namespace swab
