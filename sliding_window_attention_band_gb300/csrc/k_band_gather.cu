// k_band_gather.cu -- the two backward-mode banded products of "Developing a
// faster schedule for Longformer's kernel" (TVM forum, post 6):
//   transpose_t1 = 0 (band x dense -> dense):
//       O[i,c] = alpha * sum_t P[i,t] * V[i + (t-w)*s, c]
//   transpose_t1 = 1 (band^T x dense -> dense):
//       X[j,c] = alpha * sum over (i,t) with i + (t-w)*s = j of Bd[i,t]*Y[i,c]
// Forward P.V and dQ = dS.K use the first; dK = dS^T.Q and dV = P^T.dO the
// second.
//
// Both are run as dense tcgen05 products over a window, with the banded
// operand expanded on the fly into a dense tile in shared memory (zeros off
// the band).  The key observation: in both products one "line" of the dense
// A tile is a contiguous piece of ONE band row, shifted:
//   band_pv : A[q][k]  (M = query q, K = key k)    = P[q][k - q + const]
//   band_t  : A[m][q]  (M = key m,   K = query q)  = Bd[q][m - q + const]
// so for both the line of query q is band row q read from some slot on, and
// only the tile layout differs (K-major for band_pv, MN-major for band_t).
//
// A line starts at an arbitrary 2-byte boundary.  Lines whose query indices
// agree mod 8 start at the same offset mod 16 bytes (the row pitch in
// elements is D and the slot start moves by -1 per query), so each warp task
// takes lines of one such class: its 16-byte loads are coalesced, and the
// realignment shift is the same for all 32 lanes.  The realigned 16-byte
// pieces are written into the 128-byte-swizzled layout the tensor core reads.
//
// CTA = 128 output rows (queries for band_pv, keys for band_t) of one residue
// of the key stride; the K dimension (keys / queries) is walked 64 at a time.
// Warp 0 loads the dense operand (V or Y) with TMA, warp 1 owns tensor memory
// and issues MMAs, warps 2..9 build the A stages and finally drain the fp32
// accumulator (TMEM lane = output row).
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 4;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kBM = 128;    // output rows per tile (MMA M)
constexpr int kKC = 64;     // K per stage
// Two stages of A and B tiles (50 KB of shared memory) so that three CTAs
// share an SM (two with the global-token term, whose registers do not fit
// three): one CTA's products run while the others gather.  Four stages and
// two CTAs an SM: band_pv 37.6 / band_t 39.6 us at n = 4096, w = 256 against
// 31.4 / 33.4 us.
constexpr int kStages = 2;
constexpr int kGW = 8;      // gather warps
constexpr int kThreads = 32 * (2 + kGW);
constexpr int kATile = kBM * kKC * 2;    // 16 KB
constexpr int kBTile = kKC * 64 * 2;     // 8 KB (64 rows x 64 halves)
constexpr int kSmemBytes = kStages * (kATile + kBTile) + 1024 + 1024;
// up to this many global tokens the global term runs on the tensor cores as
// one more chunk of the pipeline (K = G rounded up to 16); beyond it, FFMA in
// the epilogue
constexpr int kGlobTc = 64;
constexpr uint32_t kTmemCols = 64;

// bytes [2e, 2e + 16) of the 32-byte value (lo, hi), e in [0, 8)
template <int E>
__device__ __forceinline__ uint4 shift_extract(const uint4 &lo, const uint4 &hi) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    constexpr int ws = E / 2;
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (E % 2 == 0) {
            o[k] = w[k + ws];
        } else {
            o[k] = __funnelshift_r(w[k + ws], w[k + ws + 1], 16);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// The same with e known only at run time (uniform across the warp).
__device__ __forceinline__ uint4 extract_elems(const uint4 &lo, const uint4 &hi, int e) {
    switch (e) {
        case 0: return lo;
        case 1: return shift_extract<1>(lo, hi);
        case 2: return shift_extract<2>(lo, hi);
        case 3: return shift_extract<3>(lo, hi);
        case 4: return shift_extract<4>(lo, hi);
        case 5: return shift_extract<5>(lo, hi);
        case 6: return shift_extract<6>(lo, hi);
        default: return shift_extract<7>(lo, hi);
    }
}

// Zero the 16-bit elements outside [lo, hi) of an 8-element piece.
__device__ __forceinline__ uint4 mask_elems(uint4 v, int lo, int hi) {
    uint32_t m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int e0 = 2 * k, e1 = 2 * k + 1;
        m[k] = ((e0 >= lo && e0 < hi) ? 0x0000ffffu : 0u) | ((e1 >= lo && e1 < hi) ? 0xffff0000u : 0u);
    }
    return make_uint4(v.x & m[0], v.y & m[1], v.z & m[2], v.w & m[3]);
}

// kUni: every gather warp's realignment shift is the same (s*D - 1 a
// multiple of 8, e.g. every undilated band with D = 2^k + 1)
template <typename T, bool kTrans, bool kGlob, bool kUni>
__global__ void __launch_bounds__(kThreads, kGlob ? 2 : 3)
    k_band_gather_tc(const __grid_constant__ TmapSet mapB, const GatherArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *atile = base;                               // kStages x 16 KB
    uint8_t *btile = base + kStages * kATile;            // kStages x 8 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(btile + kStages * kBTile);
    uint64_t *afull = bars;                  // [kStages], count kGW
    uint64_t *bfull = bars + kStages;        // [kStages], TMA
    uint64_t *empty = bars + 2 * kStages;    // [kStages], MMA commit
    uint64_t *accfull = bars + 3 * kStages;  // [1]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(accfull + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    // global tokens: a bitmap of the global positions and their dense rows
    uint32_t *gbits = reinterpret_cast<uint32_t *>(base + kStages * (kATile + kBTile) + 1024);
    float *gyrows = reinterpret_cast<float *>(gbits + (kGlob ? ((p.g.n + 31) >> 5) : 0));

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, bh = blockIdx.z;
    const int nr = residue_len(g.n, g.s, r);
    const int a0 = blockIdx.x * kBM;
    if (a0 >= nr) return;
    auto is_global = [&](long long j) -> bool {
        return kGlob && ((gbits[j >> 5] >> (j & 31)) & 1u);
    };
    // K range: keys for band_pv, queries for band_t
    const int k_lo = kTrans ? max(a0 - g.wu, 0) : max(a0 - g.w, 0);
    const int k_hi = kTrans ? min(a0 + kBM - 1 + g.w, nr - 1) : min(a0 + kBM - 1 + g.wu, nr - 1);
    const int nck = (k_hi - k_lo + kKC) / kKC;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&afull[i], kGW);
            mbar_init(&bfull[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    if constexpr (kGlob) {
        const int words = (g.n + 31) >> 5;
        for (int k = threadIdx.x; k < words; k += blockDim.x) gbits[k] = 0u;
        __syncthreads();
        for (int k = threadIdx.x; k < p.gl.G; k += blockDim.x)
            atomicOr(&gbits[p.gl.idx[k] >> 5], 1u << (p.gl.idx[k] & 31));
        if (p.gl.G > kGlobTc) {   // the FFMA epilogue's global rows of Y
            const T *ysrc = reinterpret_cast<const T *>(p.gy) + (long long)bh * g.n * 64;
            for (int e = threadIdx.x; e < p.gl.G * 64; e += blockDim.x)
                gyrows[e] = Elt<T>::to_f(*GP(g.bnd, ysrc + (long long)p.gl.idx[e >> 6] * 64 + (e & 63)));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap *mb = &mapB.m[r];
            tma_prefetch_desc(mb);
            bool okp = true;
            for (int c = 0; c < nck; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                if (!mbar_wait(&empty[st], ph ^ 1, abort_flag, p.err)) { okp = false; break; }
                mbar_arrive_expect_tx(&bfull[st], kBTile);
                tma_load_3d(btile + st * kBTile, mb, &bfull[st], 0, k_lo + c * kKC, bh);
            }
            if (kGlob && p.gl.G <= kGlobTc && okp) {
                // the global chunk: the gather warps write its B tile too
                const int st = nck % kStages;
                if (mbar_wait(&empty[st], ((nck / kStages) & 1) ^ 1, abort_flag, p.err)) mbar_arrive(&bfull[st]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t idesc = idesc_f16(kBM, 64, kBf16, kTrans, true);
            bool ok = true;
            // chunk nck (global tokens, G <= kGlobTc): the G weights of every
            // output row against the G global rows of the dense operand
            const int nall = nck + ((kGlob && p.gl.G <= kGlobTc) ? 1 : 0);
            for (int c = 0; c < nall && ok; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                ok = mbar_wait(&bfull[st], ph, abort_flag, p.err) &&
                     mbar_wait(&afull[st], ph, abort_flag, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(atile + st * kATile);
                const uint32_t b_addr = smem_u32(btile + st * kBTile);
                const int ksteps = c < nck ? kKC / 16 : (p.gl.G + 15) / 16;
#pragma unroll
                for (int k = 0; k < kKC / 16; ++k) {
                    if (k >= ksteps) break;
                    // A: K-major (band_pv) advances 32 B per K=16 step inside the
                    // 128-B swizzle row; MN-major (band_t) advances 16 lines of
                    // 128 B.  B (dense rows, MN-major) advances 16 lines.
                    const uint64_t ad = kTrans ? sdesc_sw128(a_addr + 2048 * k, kKC * 128, 1024)
                                               : sdesc_sw128(a_addr + 32 * k, 16, 1024);
                    // N = 64 is one 128-B block: the MN-block stride is unused, so it is
                    // given the same value as the 8-line K-group stride.
                    const uint64_t bd = sdesc_sw128(b_addr + 2048 * k, 1024, 1024);
                    mma_f16_ss(tmem, ad, bd, idesc, (c > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&empty[st]);
            }
            if (ok) mma_commit(accfull);
        }
    } else {
        // ---------------- gather warps ----------------
        // Each warp owns 4 of the 32 tasks of a stage (task = lines of one
        // class mod 8).  Per task the line geometry is fixed up to a per-stage
        // increment, so it is set up once; per stage the warp first issues all
        // of its band loads (up to 8 per lane, before it even waits for the
        // stage to be free), then realigns and stores them.
        const int gw = warp - 2;
        const uint16_t *band = reinterpret_cast<const uint16_t *>(p.band);
        const long long slice_row0 = (long long)bh * g.n + r;  // band row of sub-index 0
        constexpr int kTasks = 32 / kGW;
        long long e_line[kTasks];  // element offset of this lane's 8 elements, stage 0
        int vlo[kTasks];           // first valid element of the lane's piece, stage 0
        int vcap[kTasks];          // valid elements end at min(vlo + D, vcap - stage*64) (pv) / vcap (t)
        int shift[kTasks];         // realignment (the same for every task: one class mod 8)
        int qline[kTasks];         // band_t: query sub-index of the lane's line at stage 0
        int kkey[kTasks];          // key sub-index of the lane's first element at stage 0
        uint32_t dst[kTasks];      // byte offset inside the A stage
        long long e_step;          // e_line increment per stage
#pragma unroll
        for (int u = 0; u < kTasks; ++u) {
            const int task = gw + kGW * u;
            const int cls = task & 7, sub = task >> 3;
            if (!kTrans) {
                // 128 lines (queries) x 64 keys: 4 lines per task, 8 pieces each
                const int line = cls + 8 * (4 * sub + (lane >> 3));
                const int j = lane & 7;
                const int qq = a0 + line;
                const long long el = (slice_row0 + (long long)g.s * qq) * g.D + (k_lo - qq + g.w);
                shift[u] = (int)(el & 7);
                e_line[u] = el + 8 * j;
                vlo[u] = qq - g.w - k_lo - 8 * j;
                vcap[u] = (qq < nr && !is_global(r + (long long)g.s * qq)) ? (k_hi - k_lo + 1 - 8 * j)
                                                                          : -(1 << 30);
                qline[u] = 0;
                kkey[u] = k_lo + 8 * j;
                dst[u] = line * 128 + ((j ^ (line & 7)) << 4);
            } else {
                // 64 lines (queries) x 128 keys: 2 lines per task, 16 pieces each
                const int line = cls + 8 * (2 * sub + (lane >> 4));
                const int j = lane & 15;
                const int qq = k_lo + line;
                const long long el = (slice_row0 + (long long)g.s * qq) * g.D + (a0 - qq + g.w);
                shift[u] = (int)(el & 7);
                e_line[u] = el + 8 * j;
                vlo[u] = qq - g.w - a0 - 8 * j;
                vcap[u] = nr - a0 - 8 * j;
                qline[u] = qq;
                kkey[u] = a0 + 8 * j;
                dst[u] = (j >> 3) * (kKC * 128) + line * 128 + (((j & 7) ^ (line & 7)) << 4);
            }
        }
        e_step = kTrans ? (long long)kKC * ((long long)g.s * g.D - 1) : kKC;
        bool ok = true;
        // The realignment shift is the same for all of the warp's tasks and
        // stages (their lines are of one class mod 8 and a stage moves a line
        // by a multiple of 8 elements).  When it is the same for every warp
        // too (kUni), the stage loop compiled for that shift runs; otherwise
        // one loop realigns with the shift known at run time (E < 0), since
        // eight loop copies in flight on one SM would crowd its instruction
        // cache.
        auto stage_loop = [&](auto shift_c) {
        constexpr int E = decltype(shift_c)::value;

        for (int c = 0; c < nck; ++c) {
            const int st = c % kStages;
            const uint32_t ph = (c / kStages) & 1;
            uint4 lo[kTasks], hi[kTasks];
            int plo[kTasks], phi[kTasks];
#pragma unroll
            for (int u = 0; u < kTasks; ++u) {
                // valid elements of this lane's piece: [plo, phi) within [0, 8)
                int l0, h0;
                if (!kTrans) {
                    l0 = vlo[u] - kKC * c;
                    h0 = min(l0 + g.D, vcap[u] - kKC * c);
                } else {
                    l0 = vlo[u] + kKC * c;
                    const int qq = qline[u] + kKC * c;
                    h0 = (qq < nr && !is_global(r + (long long)g.s * qq)) ? min(l0 + g.D, vcap[u]) : l0;
                }
                plo[u] = max(l0, 0);
                phi[u] = min(h0, 8);
                lo[u] = make_uint4(0, 0, 0, 0);
                hi[u] = make_uint4(0, 0, 0, 0);
                if (plo[u] < phi[u]) {
                    // (kept per task for the run-time shift: one shift test per
                    // piece, not the whole loop copied per shift value)
                    const int sh = E < 0 ? shift[u] : E;
                    const uint16_t *ptr = band + (e_line[u] + e_step * c - sh);
                    if (sh + plo[u] < 8) lo[u] = ldg16(GPN(g.bnd, ptr, 16));
                    if (sh + phi[u] > 8) hi[u] = ldg16(GPN(g.bnd, ptr + 8, 16));
                }
            }
            ok = mbar_wait(&empty[st], ph ^ 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const uint32_t a_addr = smem_u32(atile + st * kATile);
#pragma unroll
            for (int u = 0; u < kTasks; ++u) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (plo[u] < phi[u]) {
                    if constexpr (E < 0) v = extract_elems(lo[u], hi[u], shift[u]);
                    else v = shift_extract<E>(lo[u], hi[u]);
                    if (plo[u] > 0 || phi[u] < 8) v = mask_elems(v, plo[u], phi[u]);
                    if constexpr (kGlob) {
                        // keys of this piece that are global are not band keys
                        const long long k0 = r + (long long)g.s * (kkey[u] + (kTrans ? 0 : kKC * c));
                        const long long k7 = k0 + 7LL * g.s;
                        if (k7 >= p.gl.idx[0] && k0 <= p.gl.idx[p.gl.G - 1]) {
                            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (is_global(k0 + (long long)e * g.s))
                                    w[e >> 1] &= (e & 1) ? 0x0000ffffu : 0xffff0000u;
                            v = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                sts16(a_addr + dst[u], v);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[st]);
        }
        };
        if constexpr (!kUni) {
            stage_loop(std::integral_constant<int, -1>{});
        } else switch (shift[0]) {
            case 0: stage_loop(std::integral_constant<int, 0>{}); break;
            case 1: stage_loop(std::integral_constant<int, 1>{}); break;
            case 2: stage_loop(std::integral_constant<int, 2>{}); break;
            case 3: stage_loop(std::integral_constant<int, 3>{}); break;
            case 4: stage_loop(std::integral_constant<int, 4>{}); break;
            case 5: stage_loop(std::integral_constant<int, 5>{}); break;
            case 6: stage_loop(std::integral_constant<int, 6>{}); break;
            default: stage_loop(std::integral_constant<int, 7>{}); break;
        }
        if (kGlob && p.gl.G <= kGlobTc && ok) {
            // the global chunk, in the layouts of a band chunk (K = global
            // index q):
            //   A  band_pv: line m (output row), W = cols[row, q];
            //      band_t: line q, the two 64-row halves 8 KB apart, W = rows[q, row]
            //   B  line q: the global row G[q] of the dense operand
            // zero past G (and, for band_pv, at a global output row)
            const int st = nck % kStages;
            const uint32_t ph = (nck / kStages) & 1;
            ok = mbar_wait(&empty[st], ph ^ 1, abort_flag, p.err);
            if (__all_sync(0xffffffffu, ok)) {
                uint8_t *at = atile + st * kATile, *bt = btile + st * kBTile;
                const int G = p.gl.G;
                const int t = gw * 32 + lane;
                const T *W = reinterpret_cast<const T *>(p.gw);
                // 16-byte chunks of 8 K indices (band_pv) or of 8 lines' rows
                // (band_t); a chunk is one 16-byte load where the weights are
                // contiguous and aligned, else it is gathered element-wise
                if (!kTrans) {
                    for (int e = t; e < kBM * 8; e += kGW * 32) {
                        const int m = e >> 3, c = e & 7, row = a0 + m;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (8 * c < G && row < nr) {
                            const long long ri = r + (long long)g.s * row;
                            if (!is_global(ri)) {
                                const T *wp = W + ((long long)bh * g.n + ri) * G + 8 * c;
                                if ((G & 7) == 0 && (reinterpret_cast<uintptr_t>(wp) & 15) == 0) {
                                    v = *GP(g.bnd, reinterpret_cast<const uint4 *>(wp));
                                } else {
                                    float f[8];
#pragma unroll
                                    for (int u = 0; u < 8; ++u) f[u] = 8 * c + u < G ? Elt<T>::to_f(*GP(g.bnd, wp + u)) : 0.f;
                                    v = make_uint4(pack2<T>(f[0], f[1]), pack2<T>(f[2], f[3]),
                                                   pack2<T>(f[4], f[5]), pack2<T>(f[6], f[7]));
                                }
                            }
                        }
                        sts16(smem_u32(at) + m * 128 + ((c ^ (m & 7)) << 4), v);
                    }
                } else {
                    for (int e = t; e < kKC * (kBM / 8); e += kGW * 32) {
                        const int q = e >> 4, m0 = 8 * (e & 15);
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (q < G) {
                            const T *wp = W + ((long long)bh * G + q) * g.n + r + (long long)g.s * (a0 + m0);
                            if (g.s == 1 && a0 + m0 + 8 <= nr &&
                                (reinterpret_cast<uintptr_t>(wp) & 15) == 0) {
                                v = *GP(g.bnd, reinterpret_cast<const uint4 *>(wp));
                            } else {
                                float f[8];
#pragma unroll
                                for (int u = 0; u < 8; ++u)
                                    f[u] = a0 + m0 + u < nr ? Elt<T>::to_f(*GP(g.bnd, wp + (long long)g.s * u)) : 0.f;
                                v = make_uint4(pack2<T>(f[0], f[1]), pack2<T>(f[2], f[3]),
                                               pack2<T>(f[4], f[5]), pack2<T>(f[6], f[7]));
                            }
                        }
                        sts16(smem_u32(at) + (m0 >> 6) * (kKC * 128) + q * 128 +
                                  ((((m0 & 63) >> 3) ^ (q & 7)) << 4), v);
                    }
                }
                const T *Y = reinterpret_cast<const T *>(p.gy) + (long long)bh * g.n * 64;
                for (int e = t; e < kKC * 8; e += kGW * 32) {
                    const int q = e >> 3, c = e & 7;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (q < G) v = *reinterpret_cast<const uint4 *>(Y + (long long)p.gl.idx[q] * 64 + 8 * c);
                    *reinterpret_cast<uint4 *>(bt + q * 128 + ((c ^ (q & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[st]);
            } else {
                ok = false;
            }
        }
        // ---------------- epilogue ----------------
        const bool acc_ok = ok && mbar_wait(accfull, 0, abort_flag, p.err);
        if (__all_sync(0xffffffffu, acc_ok)) {
            tc_fence_after();
            const int quarter = warp & 3;
            const int half = gw >> 2;  // columns [32*half, 32*half + 32)
            const int m = quarter * 32 + lane;
            uint32_t v[32];
            tmem_ld32(tmem_addr(tmem, quarter * 32, half * 32), v);
            tmem_ld_wait();
            const int row = a0 + m;
            if (kGlob && row < nr && p.gl.G > kGlobTc) {
                // band_pv: + sum_g cols[i,g] V[G[g]] for a local query row i;
                // band_t:  + sum_g rows[g,j] Y[G[g]] for key j (on FFMA here
                // past kGlobTc global tokens; up to it, the global chunk has
                // added them on the tensor cores).
                const long long ri = r + (long long)g.s * row;  // row index in the slice
                if (!kTrans && is_global(ri)) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                } else {
                    const T *gw = reinterpret_cast<const T *>(p.gw);
                    float acc[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]);
                    for (int q = 0; q < p.gl.G; ++q) {
                        const float wv = kTrans
                            ? Elt<T>::to_f(*GP(g.bnd, gw + ((long long)bh * p.gl.G + q) * g.n + ri))
                            : Elt<T>::to_f(*GP(g.bnd, gw + ((long long)bh * g.n + ri) * p.gl.G + q));
                        const float *yr = gyrows + q * 64 + half * 32;
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[i] = fmaf(wv, yr[i], acc[i]);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(acc[i]);
                }
            }
            if (kGlob && !kTrans && row < nr && p.gl.G <= kGlobTc && is_global(r + (long long)g.s * row)) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0u;   // a global query's row is dense, written apart
            }
            if (row < nr) {
                T *out = reinterpret_cast<T *>(p.out) +
                         ((long long)bh * g.n + r + (long long)g.s * row) * 64 + half * 32;
                uint4 *o4 = reinterpret_cast<uint4 *>(out);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 w;
                    w.x = pack2<T>(p.alpha * __uint_as_float(v[8 * q + 0]), p.alpha * __uint_as_float(v[8 * q + 1]));
                    w.y = pack2<T>(p.alpha * __uint_as_float(v[8 * q + 2]), p.alpha * __uint_as_float(v[8 * q + 3]));
                    w.z = pack2<T>(p.alpha * __uint_as_float(v[8 * q + 4]), p.alpha * __uint_as_float(v[8 * q + 5]));
                    w.w = pack2<T>(p.alpha * __uint_as_float(v[8 * q + 6]), p.alpha * __uint_as_float(v[8 * q + 7]));
                    *GP(g.bnd, o4 + q) = w;
                }
            }
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
// exact fp32 paths
// ---------------------------------------------------------------------------
// band_pv: one CTA per output row, one thread per channel.
__global__ void __launch_bounds__(128) k_band_pv_f32(const DenseArgs p) {
    const Geom &g = p.g;
    const long long R = blockIdx.x;
    const int i = (int)(R % g.n);
    const long long bh = R / g.n;
    const int c = threadIdx.x;
    if (c >= g.hd) return;
    const float *P = reinterpret_cast<const float *>(p.A) + R * g.D;
    const float *V = reinterpret_cast<const float *>(p.B) + bh * g.n * g.hd;
    const int t_lo = max(0, g.w - i / g.s);
    const int t_hi = min(g.D - 1, g.w + (g.n - 1 - i) / g.s);
    float acc = 0.f;
    for (int t = t_lo; t <= t_hi; ++t) {
        const long long j = (long long)i + (long long)(t - g.w) * g.s;
        acc = fmaf(*GP(g.bnd, P + t), *GP(g.bnd, V + j * g.hd + c), acc);
    }
    *GP(g.bnd, reinterpret_cast<float *>(p.out) + R * g.hd + c) = p.alpha * acc;
}

// band_t: one CTA per output row j (a key), one thread per channel; the
// queries meeting key j are i = j - (t-w)*s for the slots t that keep i in range.
__global__ void __launch_bounds__(128) k_band_t_f32(const DenseArgs p) {
    const Geom &g = p.g;
    const long long R = blockIdx.x;
    const int j = (int)(R % g.n);
    const long long bh = R / g.n;
    const int c = threadIdx.x;
    if (c >= g.hd) return;
    const float *Bd = reinterpret_cast<const float *>(p.A) + bh * g.n * g.D;
    const float *Y = reinterpret_cast<const float *>(p.B) + bh * g.n * g.hd;
    float acc = 0.f;
    for (int t = 0; t < g.D; ++t) {
        const long long i = (long long)j - (long long)(t - g.w) * g.s;
        if (i < 0 || i >= g.n) continue;
        acc = fmaf(*GP(g.bnd, Bd + i * g.D + t), *GP(g.bnd, Y + i * g.hd + c), acc);
    }
    *GP(g.bnd, reinterpret_cast<float *>(p.out) + R * g.hd + c) = p.alpha * acc;
}

template <typename T, bool kTrans, bool kGlob, bool kUni>
cudaError_t launch_gather(const TmapSet &mapB, const GatherArgs &a, cudaStream_t st) {
    const int tiles = (a.g.nsub + kBM - 1) / kBM;
    dim3 grid(tiles, a.g.s, a.g.BH);
    const size_t smem = kSmemBytes + (kGlob ? gather_glob_smem(a.g.n, a.gl.G) : 0);
    cudaError_t e =
        ensure_smem(reinterpret_cast<const void *>(k_band_gather_tc<T, kTrans, kGlob, kUni>), (int)smem);
    if (e != cudaSuccess) return e;
    k_band_gather_tc<T, kTrans, kGlob, kUni><<<grid, kThreads, smem, st>>>(mapB, a);
    return cudaGetLastError();
}

template <typename T, bool kTrans>
cudaError_t launch_gather2(const TmapSet &mapB, const GatherArgs &a, cudaStream_t st) {
    const bool uni = ((long long)a.g.s * a.g.D - 1) % 8 == 0;
    if (a.gl.G > 0)
        return uni ? launch_gather<T, kTrans, true, true>(mapB, a, st) : launch_gather<T, kTrans, true, false>(mapB, a, st);
    return uni ? launch_gather<T, kTrans, false, true>(mapB, a, st) : launch_gather<T, kTrans, false, false>(mapB, a, st);
}

}  // namespace

size_t gather_glob_smem(int n, int G) {
    return (size_t)((n + 31) / 32) * 4 + (G > kGlobTc ? (size_t)G * 64 * sizeof(float) : 0);
}

size_t gather_smem_bytes(int n, int G) { return kSmemBytes + (G > 0 ? gather_glob_smem(n, G) : 0); }

cudaError_t launch_band_gather_tc(DType dt, bool transposed, const TmapSet &mapB,
                                  const GatherArgs &a, cudaStream_t st) {
    if (dt == kF16) {
        return transposed ? launch_gather2<__half, true>(mapB, a, st)
                          : launch_gather2<__half, false>(mapB, a, st);
    }
    return transposed ? launch_gather2<__nv_bfloat16, true>(mapB, a, st)
                      : launch_gather2<__nv_bfloat16, false>(mapB, a, st);
}

cudaError_t launch_band_pv_f32(const DenseArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    k_band_pv_f32<<<(unsigned)rows, 128, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_band_t_f32(const DenseArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    k_band_t_f32<<<(unsigned)rows, 128, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace swab
