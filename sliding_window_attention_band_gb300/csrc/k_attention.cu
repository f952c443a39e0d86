// k_attention.cu -- fused forward of sliding-window attention: the same O
// (and lse) as band_qk(scale) -> band_softmax -> band_pv, with the scores
// kept on chip.  Band definition from "Developing a faster schedule for
// Longformer's kernel" (TVM forum, posts 1, 3, 6); softmax recipe (max,
// exp of the difference, sum, divide, fp32) from nvFuser issue "HuggingFace
// BertForMaskedLM - Log Softmax Fusion with Autocast has bad perf", fusion 1.
//
// One CTA = 128 query rows of one residue r of the key stride (rows
// r + s*a, a in [a0, a0+128)).  The keys its band touches are walked 128 at
// a time; for chunk c:
//   1. MMA warp: S_c = Q . K_c^T  (tcgen05, M = 128 queries, N = 128 keys,
//      K = 64) into TMEM S buffer c%2;
//   2. softmax warps (thread = query row = TMEM lane): the band is a
//      contiguous column interval of the chunk for each row (masking is two
//      compares, skipped when the whole chunk is inside every row's band).
//      Online softmax in the log2 domain with a reference max that is raised
//      only when a chunk exceeds it by more than 2^8, so each chunk is one
//      pass over tensor memory; p = 2^(x - m) rounded to fp16/bf16 is written
//      as the K-major, 128-B-swizzled A operand of the next product (smem);
//   3. MMA warp: O_c = P_c . V_c into TMEM O buffer c%2 (fresh, not
//      accumulated), split along the keys into two halves with their own
//      buffers, one per softmax warp half;
//   4. softmax warps, one chunk later (so the P.V product of chunk c runs
//      while chunk c+1's softmax is computed): acc = acc * 2^(m_prev - m) + O_c.
// At the end O = acc / l, lse = m*ln2 + ln l.
//
// Warps: 0 = TMA producer (Q once; K and V chunks into a 3-stage ring),
// 1 = TMEM owner + MMA issuer, 2..9 = softmax / epilogue (two per TMEM lane
// quarter, each owning one key half of every chunk; the halves merge their
// running max, sum and accumulator once, at the end).
#include <type_traits>

#include "swab_internal.h"

namespace swab {
namespace {

constexpr int kBQ = 128;      // queries per CTA (M)
constexpr int kBK = 128;      // keys per chunk (N of S, K of P.V)
constexpr int kStages = 3;    // K/V ring
constexpr int kThreads = 320;   // producer, MMA, 8 softmax warps (2 per TMEM lane quarter)
constexpr int kWorkers = 256;
constexpr int kQBytes = kBQ * 128;             // 16 KB
constexpr int kKBytes = kBK * 128;             // 16 KB
constexpr int kVBytes = kBK * 128;             // 16 KB
constexpr int kStageBytes = kKBytes + kVBytes; // 32 KB
constexpr int kPBytes = kBQ * kBK * 2;         // 32 KB (two 64-key K-atoms)
constexpr int kSmemBytes = kQBytes + kStages * kStageBytes + 2 * kPBytes + 1024 + 1024;
constexpr uint32_t kTmemCols = 512;            // S: 2 x 128, O: 2 chunks x 2 key halves x 64
constexpr uint32_t kTmemO = 256;               // O of chunk parity b, key half h at 256 + 128b + 64h

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    k_band_attention_fwd(const __grid_constant__ TmapSet mapQ, const __grid_constant__ TmapSet mapK,
                         const __grid_constant__ TmapSet mapV, const AttnArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qtile = base;
    uint8_t *kv = base + kQBytes;                        // stage st: K at +0, V at +kKBytes
    uint8_t *pbuf = kv + kStages * kStageBytes;          // 2 x 32 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(pbuf + 2 * kPBytes);
    uint64_t *qfull = bars;                  // 1
    uint64_t *kvfull = bars + 1;             // [kStages]
    uint64_t *kvempty = kvfull + kStages;    // [kStages]
    uint64_t *sfull = kvempty + kStages;     // [2]
    uint64_t *sempty = sfull + 2;            // [2] count 128
    uint64_t *pfull = sempty + 2;            // [2] count 128
    uint64_t *pempty = pfull + 2;            // [2]
    uint64_t *ofull = pempty + 2;            // [2]
    uint64_t *oempty = ofull + 2;            // [2] count 128
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(oempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, bh = blockIdx.z;
    const int nr = residue_len(g.n, g.s, r);
    const int a0 = blockIdx.x * kBQ;
    if (a0 >= nr) return;
    const int kb_lo = max(a0 - g.w, 0);
    const int kb_hi = min(a0 + kBQ - 1 + g.wu, nr - 1);
    const int nck = (kb_hi - kb_lo + kBK) / kBK;

    if (threadIdx.x == 0) {
        mbar_init(qfull, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], kWorkers);
            mbar_init(&pfull[i], kWorkers);
            mbar_init(&pempty[i], 1);
            mbar_init(&ofull[i], 1);
            mbar_init(&oempty[i], kWorkers);
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
            const CUtensorMap *mq = &mapQ.m[r], *mk = &mapK.m[r], *mv = &mapV.m[r];
            tma_prefetch_desc(mq);
            tma_prefetch_desc(mk);
            tma_prefetch_desc(mv);
            mbar_arrive_expect_tx(qfull, kQBytes);
            tma_load_3d(qtile, mq, qfull, 0, a0, bh);
            for (int c = 0; c < nck; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                if (!mbar_wait(&kvempty[st], ph ^ 1, abort_flag, p.err)) break;
                mbar_arrive_expect_tx(&kvfull[st], kStageBytes);
                uint8_t *stage = kv + st * kStageBytes;
                tma_load_3d(stage, mk, &kvfull[st], 0, kb_lo + c * kBK, bh);
                tma_load_3d(stage + kKBytes, mv, &kvfull[st], 0, kb_lo + c * kBK, bh);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t idesc_s = idesc_f16(kBQ, kBK, kBf16, false, false);
            const uint32_t idesc_o = idesc_f16(kBQ, 64, kBf16, false, true);
            const uint32_t q_addr = smem_u32(qtile);
            bool ok = mbar_wait(qfull, 0, abort_flag, p.err);
            // P.V of chunk c (issued after S of chunk c+1 so that the two overlap)
            auto issue_pv = [&](int c) -> bool {
                const int st = c % kStages;
                const int b = c & 1;
                const uint32_t bph = (c >> 1) & 1;
                if (!mbar_wait(&pfull[b], bph, abort_flag, p.err)) return false;
                if (!mbar_wait(&oempty[b], bph ^ 1, abort_flag, p.err)) return false;
                tc_fence_after();
                const uint32_t p_addr = smem_u32(pbuf + b * kPBytes);
                const uint32_t v_addr = smem_u32(kv + st * kStageBytes + kKBytes);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // keys [64h, 64h + 64): K-atom h of P, rows 64h.. of V
                    const uint32_t d = tmem + kTmemO + b * 128 + h * 64;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t a = p_addr + h * (kPBytes / 2) + k * 32;
                        mma_f16_ss(d, sdesc_sw128(a, 16, 1024),
                                   sdesc_sw128(v_addr + h * 8192 + 2048 * k, 1024, 1024), idesc_o, k > 0);
                    }
                }
                mma_commit(&ofull[b]);
                mma_commit(&pempty[b]);
                mma_commit(&kvempty[st]);
                return true;
            };
            for (int c = 0; c < nck && ok; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                const int b = c & 1;
                const uint32_t bph = (c >> 1) & 1;
                ok = mbar_wait(&kvfull[st], ph, abort_flag, p.err) &&
                     mbar_wait(&sempty[b], bph ^ 1, abort_flag, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(kv + st * kStageBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    mma_f16_ss(tmem + b * kBK, sdesc_sw128(q_addr + 32 * k, 16, 1024),
                               sdesc_sw128(k_addr + 32 * k, 16, 1024), idesc_s, k > 0);
                }
                mma_commit(&sfull[b]);
                if (c > 0) ok = issue_pv(c - 1);
            }
            if (ok) issue_pv(nck - 1);
        }
    } else {
        // ---------------- softmax warps: thread = query row ----------------
        // Two warps per TMEM lane quarter: warp half h owns key columns
        // [64h, 64h + 64) of every chunk and keeps its own reference max m,
        // sum l and accumulator (its P.V half goes to its own TMEM buffer), so
        // the halves never wait on each other until the final merge.
        // Per half: a chunk is processed in ONE pass over tensor memory with
        // the current m; m is raised only when the chunk's largest score
        // exceeds it by more than kSlack (the chunk is then redone with the
        // new m), so p <= 2^kSlack stays well inside fp16/bf16 range.  A half
        // with no key seen yet takes its m from a max-only pass first.  The
        // softmax does not depend on the choice of m.
        constexpr float kSlack = 8.f;
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int q = quarter * 32 + lane;
        const int qq = a0 + q;
        const float xscale = p.scale * 1.4426950408889634f;
        float m = -INFINITY, l = 0.f, corr_prev = 1.f;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.f;
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        bool ok = true;

        auto fold_o = [&](int c, float corr) -> bool {
            const int b = c & 1;
            const uint32_t bph = (c >> 1) & 1;
            const bool w_ok = mbar_wait(&ofull[b], bph, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) return false;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v[32];
                tmem_ld32(lane_base + kTmemO + b * 128 + half * 64 + h * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[h * 32 + i] = fmaf(acc[h * 32 + i], corr, __uint_as_float(v[i]));
            }
            tc_fence_before();
            mbar_arrive(&oempty[b]);
            return true;
        };

        for (int c = 0; c < nck; ++c) {
            const int b = c & 1;
            const uint32_t bph = (c >> 1) & 1;
            const int kbase = kb_lo + c * kBK;
            // this row's band inside the chunk: columns [jlo, jhi]
            const int jlo = max(qq - g.w - kbase, 0);
            const int jhi = min(min(qq + g.wu, kb_hi) - kbase, kBK - 1);
            const bool full = __all_sync(0xffffffffu, jlo <= 64 * half && jhi >= 64 * half + 63);
            bool w_ok = mbar_wait(&sfull[b], bph, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sbuf = lane_base + b * kBK;
            float mref = m;
            if (__any_sync(0xffffffffu, m == -INFINITY)) {
                float mx = -INFINITY;
#pragma unroll 1
                for (int grp = 2 * half; grp < 2 * half + 2; ++grp) {
                    uint32_t v[32];
                    tmem_ld32(sbuf + grp * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = grp * 32 + i;
                        if (j >= jlo && j <= jhi) mx = fmaxf(mx, __uint_as_float(v[i]) * xscale);
                    }
                }
                if (m == -INFINITY) mref = mx;
            }
            // the P tile of chunk c may still feed the P.V product of chunk c-2
            w_ok = mbar_wait(&pempty[b], bph ^ 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
            const uint32_t pbase = smem_u32(pbuf + b * kPBytes);
            float lc = 0.f;
            for (int pass = 0; pass < 2; ++pass) {
                const float mb = mref == -INFINITY ? 0.f : mref;
                float ymax = -INFINITY;  // chunk max relative to mref
                lc = 0.f;
#pragma unroll 1
                for (int grp = 2 * half; grp < 2 * half + 2; ++grp) {
                    uint32_t v[32];
                    tmem_ld32(sbuf + grp * 32, v);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float y0 = fmaf(__uint_as_float(v[2 * i]), xscale, -mb);
                        float y1 = fmaf(__uint_as_float(v[2 * i + 1]), xscale, -mb);
                        if (!full) {
                            const int j0 = grp * 32 + 2 * i;
                            if (j0 < jlo || j0 > jhi) y0 = -INFINITY;
                            if (j0 + 1 < jlo || j0 + 1 > jhi) y1 = -INFINITY;
                        }
                        ymax = fmaxf(ymax, fmaxf(y0, y1));
                        const float p0 = ex2(y0), p1 = ex2(y1);
                        lc += p0 + p1;
                        pk[i] = pack2<T>(p0, p1);
                    }
                    // 32 keys = 4 x 16-byte pieces; key-atom grp/2, pieces (grp%2)*4 + 0..3
                    const uint32_t atom = pbase + (grp >> 1) * (kPBytes / 2) + q * 128;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int piece = (grp & 1) * 4 + u;
                        sts16(atom + ((piece ^ (q & 7)) << 4),
                              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
                    }
                }
                // redo the chunk if a score rose more than kSlack above mref
                const bool redo = ymax > kSlack;
                if (!__any_sync(0xffffffffu, redo)) break;
                if (redo) mref = mb + ymax;
            }
            const float corr = (m == -INFINITY) ? 1.f : ex2(m - mref);
            l = l * corr + lc;
            tc_fence_before();
            mbar_arrive(&sempty[b]);   // S buffer b may be overwritten
            fence_proxy_async_smem();
            mbar_arrive(&pfull[b]);    // P tile b is ready for the tensor core
            m = mref;
            if (c > 0) {
                if (!fold_o(c - 1, corr_prev)) { ok = false; break; }
            }
            corr_prev = corr;
        }
        if (ok) ok = fold_o(nck - 1, corr_prev);
        // merge the two key halves: every P.V product is complete, so the P
        // tiles are free to carry each half's (m, l) and the accumulator
        // channels the other half writes out
        float *xs = reinterpret_cast<float *>(pbuf);  // [2 halves][128 rows][34]
        const bool all_ok = __all_sync(0xffffffffu, ok);
        // static register indices only: split acc by half with branches
        float keep[32], give[32];
        if (half == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                keep[i] = acc[i];
                give[i] = acc[32 + i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                keep[i] = acc[32 + i];
                give[i] = acc[i];
            }
        }
        if (all_ok) {
            float *mine = xs + (half * kBQ + q) * 34;
            mine[0] = m;
            mine[1] = l;
#pragma unroll
            for (int i = 0; i < 32; ++i) mine[2 + i] = give[i];
        }
        named_bar_sync(1, kWorkers);
        if (all_ok && qq < nr) {
            const float *other = xs + ((1 - half) * kBQ + q) * 34;
            const float pm = other[0], pl = other[1];
            const float M = fmaxf(m, pm);
            const float f = m == -INFINITY ? 0.f : ex2(m - M);
            const float pf = pm == -INFINITY ? 0.f : ex2(pm - M);
            const float inv = 1.f / (l * f + pl * pf);
            T *out = reinterpret_cast<T *>(p.O) + ((long long)bh * g.n + r + (long long)g.s * qq) * 64 +
                     half * 32;
            uint4 *o4 = reinterpret_cast<uint4 *>(out);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    y[e] = (keep[8 * u + e] * f + other[2 + 8 * u + e] * pf) * inv;
                o4[u] = make_uint4(pack2<T>(y[0], y[1]), pack2<T>(y[2], y[3]), pack2<T>(y[4], y[5]),
                                   pack2<T>(y[6], y[7]));
            }
            if (p.lse && half == 0)
                p.lse[(long long)bh * g.n + r + (long long)g.s * qq] =
                    M * 0.6931471805599453f + logf(l * f + pl * pf);
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
// exact fp32 path: one CTA per query row, one thread per channel; each band
// slot's score is a block-wide dot product, folded into an online softmax.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_band_attention_f32(const AttnArgsF32 p) {
    const Geom &g = p.g;
    const long long R = blockIdx.x;
    const int i = (int)(R % g.n);
    const long long bh = R / g.n;
    const int c = threadIdx.x;
    const int lane = c & 31, wid = c >> 5, nw = (blockDim.x + 31) >> 5;
    __shared__ float part[4];
    const float *Q = p.Q + R * g.hd;
    const float *K = p.K + bh * g.n * g.hd;
    const float *V = p.V + bh * g.n * g.hd;
    const float qc = c < g.hd ? Q[c] : 0.f;
    const int t_lo = max(0, g.w - i / g.s);
    const int t_hi = min(g.D - 1, g.w + (g.n - 1 - i) / g.s);
    float m = -INFINITY, l = 0.f, acc = 0.f;
    for (int t = t_lo; t <= t_hi; ++t) {
        const long long j = (long long)i + (long long)(t - g.w) * g.s;
        float x = c < g.hd ? qc * K[j * g.hd + c] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) part[wid] = x;
        __syncthreads();
        float sdot = 0.f;
        for (int k = 0; k < nw; ++k) sdot += part[k];
        __syncthreads();
        const float sc = sdot * p.scale;
        const float m_new = fmaxf(m, sc);
        const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
        const float pv = expf(sc - m_new);
        l = l * corr + pv;
        if (c < g.hd) acc = acc * corr + pv * V[j * g.hd + c];
        m = m_new;
    }
    if (c < g.hd) p.O[R * g.hd + c] = acc / l;
    if (c == 0 && p.lse) p.lse[R] = m + logf(l);
}

template <typename T>
cudaError_t launch_t(const TmapSet &mq, const TmapSet &mk, const TmapSet &mv, const AttnArgs &a,
                     cudaStream_t st) {
    const int tiles = (a.g.nsub + kBQ - 1) / kBQ;
    dim3 grid(tiles, a.g.s, a.g.BH);
    cudaError_t e = cudaFuncSetAttribute(k_band_attention_fwd<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    k_band_attention_fwd<T><<<grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band_attention_f32(const AttnArgsF32 &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    const int threads = ((a.g.hd + 31) / 32) * 32;
    k_band_attention_f32<<<(unsigned)rows, threads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_band_attention_tc(DType dt, const TmapSet &mapQ, const TmapSet &mapK,
                                     const TmapSet &mapV, const AttnArgs &a, cudaStream_t st) {
    if (dt == kF16) return launch_t<__half>(mapQ, mapK, mapV, a, st);
    return launch_t<__nv_bfloat16>(mapQ, mapK, mapV, a, st);
}

}  // namespace swab
