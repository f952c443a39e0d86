// k_attention.cu -- fused forward of sliding-window attention: the same O
// (and lse) as band_qk(scale) -> band_softmax -> band_pv, with the scores
// kept on chip.  Band definition from "Developing a faster schedule for
// Longformer's kernel" (TVM forum, posts 1, 3, 6); softmax recipe (max,
// exp of the difference, sum, divide, fp32) from nvFuser issue "HuggingFace
// BertForMaskedLM - Log Softmax Fusion with Autocast has bad perf", fusion 1.
//
// Work unit ("tile") = 128 query rows of one residue r of the key stride
// (rows r + s*a, a in [a0, a0+128)).  The kernel is persistent: one CTA per
// SM walks the tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...; a per-CTA
// chunk counter runs across tiles, so the K/V ring, the score and P buffers
// and their barriers carry straight on from one tile into the next.  For
// chunk c (128 keys) of a tile, with b = c mod 2:
//   1. MMA thread: S_b = Q . K_c^T (tcgen05, M = 128 queries, N = 128 keys,
//      K = 64) into tensor-memory score buffer b;
//   2. softmax warps, two per TMEM lane quarter: the warp of half h owns keys
//      [64h, 64h+64) of the chunk for its 32 query rows (thread = row).  It
//      copies its 64 scores to registers (which frees S_b for chunk c+2),
//      applies the band as per-32-key masks (warp-uniform fast paths for
//      groups that are full or empty for the whole warp), takes the max and
//      p = 2^(x*scale*log2e - m_h) with packed fp32x2 arithmetic and ex2,
//      and packs p to 16 bits into its 32 columns of the tensor-memory P
//      buffer b.  Each half keeps its own reference max m_h and sum l_h, and
//      raises m_h only when a chunk's largest score exceeds it by more than
//      2^8 (p <= 2^8 stays inside fp16 / bf16); its accumulator rows are
//      rescaled in place then (rare);
//   3. MMA thread: O_h += P_b[:, half h] . V_c[half h] for h = 0, 1 (A read
//      from tensor memory, B = V rows from shared memory, N = 64) into the
//      half's own fp32 accumulator.
// S and P are double-buffered, so a chunk's softmax overlaps the next
// chunk's Q.K^T and the previous chunk's P.V; nothing waits for the previous
// P.V except a rescale and the tile's epilogue.  The epilogue (in the next
// tile's first chunk, after its P is written and before it is signalled)
// exchanges (m_h, l_h) between the two halves of a row through shared memory
// and writes O = sum_h 2^(m_h - M) O_h / sum_h 2^(m_h - M) l_h, each half 32
// channels, and lse = M ln 2 + ln L.
//
// Warps: 0 = TMA producer (Q double-buffered, K and V chunks into a 4-stage
// ring), 1 = TMEM owner + MMA issuer, 2..9 = softmax / epilogue.  In the
// producer and MMA warps one lane does the work and the others go straight
// to the final barrier.  (The two roles do not share a warp: a lane spinning
// on a barrier starves a diverged lane of the same warp.)  Every wait is a
// bounded mbarrier wait (no bar.sync inside the loops), so a timeout
// anywhere lets every thread leave.
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 1;   // site id of the bounds checks

namespace swab {
namespace {

constexpr int kBQ = 128;        // queries per tile (M)
constexpr int kBK = 128;        // keys per chunk (N of S, K of P.V)
constexpr int kHalf = 64;       // keys of a chunk per softmax thread
constexpr int kStages = 4;      // K/V ring
constexpr int kWorkerWarps = 8; // two per TMEM lane quarter
constexpr int kWorkers = 32 * kWorkerWarps;     // 256
constexpr int kThreads = 64 + kWorkers;         // producer, MMA, softmax warps
constexpr int kTileBytes = kBQ * 128;           // 16 KB: 128 rows x 64 16-bit values
constexpr int kStageBytes = 2 * kTileBytes;     // K and V of a chunk
constexpr int kMlBytes = 2 * 2 * kBQ * 8;       // (m, l) exchange, two tile parities x two halves
constexpr int kBiasBytes = kWorkerWarps * kHalf * 4;   // each softmax warp's key bias of a chunk
constexpr int kBarBytes = 256;
constexpr int kSmemBytes = 2 * kTileBytes + kStages * kStageBytes + kMlBytes + kBiasBytes + kBarBytes + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S_b at 128 b
constexpr uint32_t kColP = 256;   // P_b at 256 + 64 b (half h at + 32 h)
constexpr uint32_t kColO = 384;   // O_h at 384 + 64 h
constexpr float kSlack = 8.f;     // log2 headroom of the reference max
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Largest (kMin: smallest) of the 32 values v[0..31] (fp32 bit patterns):
// four independent chains of three-input max.
template <bool kMin>
__device__ __forceinline__ float reduce32(const uint32_t *v) {
    float c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t *y = v + 8 * k;
#define F(i) __uint_as_float(y[i])
        float a = kMin ? min3(F(0), F(1), F(2)) : max3(F(0), F(1), F(2));
        a = kMin ? min3(a, F(3), F(4)) : max3(a, F(3), F(4));
        a = kMin ? min3(a, F(5), F(6)) : max3(a, F(5), F(6));
        c[k] = kMin ? fminf(a, F(7)) : fmaxf(a, F(7));
#undef F
    }
    return kMin ? fminf(min3(c[0], c[1], c[2]), c[3]) : fmaxf(max3(c[0], c[1], c[2]), c[3]);
}

struct Tile {
    int a0, r, bh, nr, kb_lo, kb_hi, nck;
};

// Tile t -> (query block, residue, slice); false when the block lies past the
// end of its residue (every role skips such tiles the same way).
__device__ __forceinline__ bool decode_tile(const Geom &g, int t, int xt, Tile &tl) {
    tl.a0 = (t % xt) * kBQ;
    const int rest = t / xt;
    tl.r = rest % g.s;
    tl.bh = rest / g.s;
    tl.nr = residue_len(g.n, g.s, tl.r);
    if (tl.a0 >= tl.nr) return false;
    // the key range starts on a multiple of 32 (keys before the band are
    // masked), so each 32-key group of a chunk is one dropout block
    tl.kb_lo = max(tl.a0 - g.w, 0) & ~31;
    tl.kb_hi = min(tl.a0 + kBQ - 1 + g.wu, tl.nr - 1);
    tl.nck = (tl.kb_hi - tl.kb_lo + kBK) / kBK;
    return true;
}

template <typename T, bool kBias, bool kDrop, bool kGlob>
__global__ void __launch_bounds__(kThreads, 1)
    k_band_attention_fwd(const __grid_constant__ TmapSet mapQ, const __grid_constant__ TmapSet mapK,
                         const __grid_constant__ TmapSet mapV, const AttnArgs p,
                         const __grid_constant__ GlobArgs gl) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qtile = base;                                   // [2] x 16 KB
    uint8_t *kv = qtile + 2 * kTileBytes;                    // stage st: K at +0, V at +kTileBytes
    float2 *mlx = reinterpret_cast<float2 *>(kv + kStages * kStageBytes);   // [2 parities][2 halves][kBQ]
    float *bslots = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(mlx) + kMlBytes);  // [8 warps][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(bslots) + kBiasBytes);
    uint64_t *qfull = bars;                  // [2]
    uint64_t *qempty = qfull + 2;            // [2]
    uint64_t *kvfull = qempty + 2;           // [kStages]
    uint64_t *kvempty = kvfull + kStages;    // [kStages]
    uint64_t *sfull = kvempty + kStages;     // [2]: S_b is in TMEM
    uint64_t *sempty = sfull + 2;            // [2], one arrival per softmax warp: S_b copied to registers
    uint64_t *pfull = sempty + 2;            // [2], one arrival per softmax warp: P_b (and a rescaled O) in TMEM
    uint64_t *pempty = pfull + 2;            // [2]: the P.V product that read P_b is done
    uint64_t *mlbar = pempty + 2;            // [4] per lane quarter, one arrival per warp (2)
    uint64_t *mmadone = mlbar + 4;           // 1: drain of the MMA pipe at exit
    uint64_t *drain = mmadone + 1;           // 1 int: never set (drain waits ignore aborts)
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(drain);
    // global tokens: bit j of gbits marks position j as global (the band
    // excludes those keys; they are attended through their own columns)
    uint32_t *gbits = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(bars) + kBarBytes);

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int xt = (g.nsub + kBQ - 1) / kBQ;
    const int ntiles = xt * g.s * g.BH;

    if constexpr (kGlob) {
        for (int w = threadIdx.x; w < (g.n + 31) / 32; w += kThreads) gbits[w] = 0u;
        __syncthreads();
        for (int k = threadIdx.x; k < gl.G; k += kThreads)
            atomicOr(&gbits[gl.idx[k] >> 5], 1u << (gl.idx[k] & 31));
        // visible to every thread after the barrier below
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], kWorkers / 32);   // one arrival per softmax warp
            mbar_init(&pfull[i], kWorkers / 32);
            mbar_init(&pempty[i], 1);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&mlbar[i], 2);   // the two warps of a lane quarter
        mbar_init(mmadone, 1);
        *no_abort = 0;
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

    if (warp == 0 && lane == 0) {
        uint32_t gc = 0, it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            Tile tl;
            if (!decode_tile(g, t, xt, tl)) continue;
            const CUtensorMap *mq = &mapQ.m[tl.r], *mk = &mapK.m[tl.r], *mv = &mapV.m[tl.r];
            const int qb = it & 1;
            if (!mbar_wait(&qempty[qb], ((it >> 1) & 1) ^ 1, abort_flag, p.err)) break;
            tma_prefetch_desc(mq);
            tma_prefetch_desc(mk);
            tma_prefetch_desc(mv);
            mbar_arrive_expect_tx(&qfull[qb], kTileBytes);
            tma_load_dense(qtile + qb * kTileBytes, mq, &qfull[qb], tl.a0, tl.bh, g.h, g.rs_p != 0);
            ++it;
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int st = gc % kStages;
                if (!mbar_wait(&kvempty[st], ((gc / kStages) & 1) ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                uint8_t *stage = kv + st * kStageBytes;
                const int row = tl.kb_lo + c * kBK;
                mbar_arrive_expect_tx(&kvfull[st], kStageBytes);
                tma_load_dense(stage, mk, &kvfull[st], row, tl.bh, g.h, g.rs_p != 0);
                tma_load_dense(stage + kTileBytes, mv, &kvfull[st], row, tl.bh, g.h, g.rs_p != 0);
            }
        }
        // every copy issued lands before the CTA may exit (the last use of
        // each stage and Q buffer; earlier ones completed before reuse)
        for (uint32_t k = gc > (uint32_t)kStages ? gc - kStages : 0; k < gc; ++k)
            mbar_wait(&kvfull[k % kStages], (k / kStages) & 1, no_abort, nullptr, 100000000ull);
        for (uint32_t k = it > 2u ? it - 2 : 0; k < it; ++k)
            mbar_wait(&qfull[k & 1], (k >> 1) & 1, no_abort, nullptr, 100000000ull);
    } else if (warp == 1 && lane == 0) {
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        constexpr uint32_t idesc_s = idesc_f16(kBQ, kBK, kBf16, false, false);
        constexpr uint32_t idesc_o = idesc_f16(kBQ, 64, kBf16, false, true);
        // Shared-memory descriptors are built once; a buffer, stage or K step
        // only moves the start address field (address >> 4, below 2^14 for any
        // shared-memory address), so each one is a 64-bit add.
        const uint64_t qdesc = sdesc_sw128(smem_u32(qtile), 16, 1024);
        const uint64_t kdesc = sdesc_sw128(smem_u32(kv), 16, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(kv + kTileBytes), 1024, 1024);
        // O_h (+)= P_b[:, half h] . V[half h], the product of chunk gg: per
        // half 4 steps of 16 keys, A from tensor memory (8 columns a step), B
        // = 16 V rows (MN-major, 2 KB a step)
        auto issue_pv = [&](uint32_t gg, bool first) -> bool {
            const int st = gg % kStages;
            const int b = gg & 1;
            if (!mbar_wait(&pfull[b], (gg >> 1) & 1, abort_flag, p.err)) return false;
            tc_fence_after();
            const uint64_t va = vdesc + (uint64_t)((st * kStageBytes) >> 4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int k = 0; k < kHalf / 16; ++k)
                    mma_f16_ts(tmem + kColO + 64 * h, tmem + kColP + 64 * b + 32 * h + 8 * k,
                               va + (uint64_t)((2048 * (4 * h + k)) >> 4), idesc_o, (first && k == 0) ? 0u : 1u);
            }
            mma_commit(&pempty[b]);
            mma_commit(&kvempty[st]);
            return true;
        };
        uint32_t gc = 0, it = 0, prev = 0;
        bool ok = true, have_prev = false, prev_first = false;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            Tile tl;
            if (!decode_tile(g, t, xt, tl)) continue;
            const int qb = it & 1;
            if (!mbar_wait(&qfull[qb], (it >> 1) & 1, abort_flag, p.err)) {
                ok = false;
                break;
            }
            const uint64_t qa = qdesc + (uint64_t)((qb * kTileBytes) >> 4);
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int st = gc % kStages;
                const int b = gc & 1;
                ok = mbar_wait(&kvfull[st], (gc / kStages) & 1, abort_flag, p.err) &&
                     mbar_wait(&sempty[b], ((gc >> 1) & 1) ^ 1, abort_flag, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ka = kdesc + (uint64_t)((st * kStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_f16_ss(tmem + kColS + kBK * b, qa + 2 * k, ka + 2 * k, idesc_s, k > 0);
                if (c == tl.nck - 1) mma_commit(&qempty[qb]);
                mma_commit(&sfull[b]);
                if (have_prev && !issue_pv(prev, prev_first)) {
                    ok = false;
                    break;
                }
                have_prev = true;
                prev = gc;
                prev_first = c == 0;
            }
            ++it;
        }
        if (ok && have_prev) issue_pv(prev, prev_first);
        // every product issued is complete before the accumulators are freed
        mma_commit(mmadone);
        mbar_wait(mmadone, 0, no_abort, nullptr, 100000000ull);
    } else if (warp >= 2) {
        // ---------------- softmax warps: thread = query row, half h of the keys ----------------
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int q = quarter * 32 + lane;
        const float xscale = p.scale * kLog2e;
        const bool neg_scale = xscale < 0.f;
        const float dscale = 256.f / (256.f - (float)g.drop_t);   // kept values' scale
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        const uint32_t o_mine = lane_base + kColO + 64 * half;
        float *bslot = bslots + (warp - 2) * kHalf;
        uint32_t gc = 0, it = 0;
        bool ok = true;
        bool epi_pend = false, epi_ok = false;
        float epi_m = 0.f, epi_l = 0.f;
        long long epi_row = 0;
        uint32_t epi_it = 0;
        // the epilogue of tile epi_it (row epi_row, this half's (epi_m, epi_l));
        // the caller has waited for the tile's last P.V product
        auto epilogue = [&]() -> bool {
            epi_pend = false;
            float2 *ml = mlx + (epi_it & 1) * 2 * kBQ;
            ml[half * kBQ + q] = make_float2(epi_m, epi_l);
            mbar_arrive_warp(&mlbar[quarter]);
            if (!__all_sync(0xffffffffu, mbar_wait(&mlbar[quarter], epi_it & 1, abort_flag, p.err)))
                return false;
            const float2 e0 = ml[q], e1 = ml[kBQ + q];
            const float M = fmaxf(e0.x, e1.x);
            const float f0 = e0.x == -INFINITY ? 0.f : ex2(e0.x - M);
            const float f1 = e1.x == -INFINITY ? 0.f : ex2(e1.x - M);
            const float L = e0.y * f0 + e1.y * f1;
            const float inv = (kDrop ? dscale : 1.f) / L;   // kept values scaled once, here
            const float g0 = f0 * inv, g1 = f1 * inv;
            // channels [32 half, 32 half + 32) of both accumulators, 16 at a time
            uint4 *o4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.O) + dense_row(g, epi_row, g.rs_o) +
                                                  32 * half);
#pragma unroll 1
            for (int v = 0; v < 2; ++v) {
                uint32_t o0[16], o1[16];
                tmem_ld16(lane_base + kColO + 32 * half + 16 * v, o0);
                tmem_ld16(lane_base + kColO + 64 + 32 * half + 16 * v, o1);
                tmem_ld_wait();
                if (epi_ok) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 8 * u + 2 * e;
                            w4[e] = pack2<T>(fmaf(__uint_as_float(o1[i]), g1, __uint_as_float(o0[i]) * g0),
                                             fmaf(__uint_as_float(o1[i + 1]), g1, __uint_as_float(o0[i + 1]) * g0));
                        }
                        *GP(g.bnd, &o4[2 * v + u]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            if (epi_ok) {
                if (p.lse && half == 0) *GP(g.bnd, p.lse + epi_row) = M * 0.6931471805599453f + logf(L);
            }
            return true;
        };
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            Tile tl;
            if (!decode_tile(g, t, xt, tl)) continue;
            const int qq = tl.a0 + q;
            float m = -INFINITY, l = 0.f;
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int b = gc & 1;
                const int kbase = tl.kb_lo + c * kBK + kHalf * half;   // this half's first key
                // this row's band inside the half: columns [jlo, jhi]
                const int jlo = qq - g.w - kbase;
                const int jhi = min(qq + g.wu, tl.kb_hi) - kbase;
                // group gi (keys kbase + 32 gi ..) is full / empty for every row
                // of the warp (rows wq0 .. wq0 + 31): warp-uniform, no vote
                const int wq0 = tl.a0 + 32 * quarter;
                const int wlo_last = wq0 + 31 - g.w - kbase;                 // largest jlo of the warp
                const int whi_first = min(wq0 + g.wu, tl.kb_hi) - kbase;    // smallest jhi
                const int wlo_first = wq0 - g.w - kbase;                     // smallest jlo
                const int whi_last = min(wq0 + 31 + g.wu, tl.kb_hi) - kbase; // largest jhi
                uint32_t vm[2];
                bool gfull[2], gempty[2];
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    gfull[gi] = wlo_last <= 32 * gi && whi_first >= 32 * gi + 31;
                    gempty[gi] = whi_last < 32 * gi || wlo_first > 32 * gi + 31;
                    const int lo = max(jlo - 32 * gi, 0), hi = min(jhi - 32 * gi, 31);
                    vm[gi] = lo > hi ? 0u : ((2u << hi) - 1u) & (0xffffffffu << lo);
                    if constexpr (kGlob) {
                        // key `lane` of the group is kbase + 32 gi + lane of the residue
                        const int sub = kbase + 32 * gi + lane;
                        const int key = tl.r + g.s * sub;
                        const bool isg = sub < tl.nr && ((gbits[key >> 5] >> (key & 31)) & 1u);
                        const uint32_t gm = __ballot_sync(0xffffffffu, isg);
                        vm[gi] &= ~gm;
                        if (gm != 0u) gfull[gi] = false;   // the masks then drop the global keys
                    }
                }
                // dropout keep bits of this row's keys, one Philox block per group
                uint32_t keep[2] = {0xffffffffu, 0xffffffffu};
                if constexpr (kDrop) {
#pragma unroll
                    for (int gi = 0; gi < 2; ++gi) {
                        if (vm[gi] != 0u && qq < tl.nr) {
                            unsigned long long wv[4];
                            philox4x64_10((unsigned long long)((kbase + 32 * gi) / 32),
                                          (unsigned long long)(tl.r + (long long)g.s * qq),
                                          (unsigned long long)tl.bh, 0, g.seed, 0, wv);
                            keep[gi] = keep_bits32(wv, g.drop_t);
                            if (g.dmask) {   // the keep-bit cache the backward reads
                                const long long wi =
                                    dmask_word(g, tl.bh, tl.r + (long long)g.s * qq, qq, (kbase + 32 * gi) / 32);
                                if (wi >= 0) *GP(g.bnd, g.dmask + wi) = keep[gi];
                            }
                        }
                    }
                }
                if constexpr (kBias) {
                    // the half's key bias (log2 units) into this warp's slot
                    __syncwarp();   // the previous chunk's reads of the slot are done
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int sub = kbase + 32 * u + lane;
                        float kb = 0.f;
                        if (!gempty[u] && sub < tl.nr)
                            kb = __ldg(GP(g.bnd, g.kbias + (size_t)(tl.bh / g.h) * g.n + tl.r + (size_t)g.s * sub)) * kLog2e;
                        bslot[32 * u + lane] = kb;
                    }
                    __syncwarp();
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&sfull[b], (gc >> 1) & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t x[kHalf];
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    if (gempty[gi]) continue;
                    uint32_t (&xg)[32] = *reinterpret_cast<uint32_t (*)[32]>(x + 32 * gi);
                    tmem_ld32(lane_base + kColS + kBK * b + kHalf * half + 32 * gi, xg);
                }
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive_warp(&sempty[b]);   // the scores are in registers: S_b may be rewritten
                const bool neg = kBias ? false : neg_scale;
                const float never = neg ? INFINITY : -INFINITY;   // the masked value that never wins
                float ext = never;
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    if (gempty[gi]) continue;
                    uint32_t *xg = x + 32 * gi;
                    if constexpr (kBias) {
                        // scaled score plus the key bias, in log2 units: the
                        // passes below see scale 1
                        const float4 *b4 = reinterpret_cast<const float4 *>(bslot + 32 * gi);
                        const uint64_t xs2 = f2(xscale, xscale);
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const float4 bb = b4[u];
                            float y0, y1, y2, y3;
                            f2split(fma2(f2(__uint_as_float(xg[4 * u]), __uint_as_float(xg[4 * u + 1])), xs2,
                                         f2(bb.x, bb.y)), y0, y1);
                            f2split(fma2(f2(__uint_as_float(xg[4 * u + 2]), __uint_as_float(xg[4 * u + 3])), xs2,
                                         f2(bb.z, bb.w)), y2, y3);
                            xg[4 * u] = __float_as_uint(y0);
                            xg[4 * u + 1] = __float_as_uint(y1);
                            xg[4 * u + 2] = __float_as_uint(y2);
                            xg[4 * u + 3] = __float_as_uint(y3);
                        }
                    }
                    if (!gfull[gi]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (!((vm[gi] >> i) & 1u)) xg[i] = __float_as_uint(never);
                    }
                    ext = neg ? fminf(ext, reduce32<true>(xg)) : fmaxf(ext, reduce32<false>(xg));
                }
                const float cmax = (vm[0] | vm[1]) != 0u ? ext * (kBias ? 1.f : xscale) : -INFINITY;
                const bool raise = m == -INFINITY || cmax > m + kSlack;
                const float mref = raise ? cmax : m;
                const float mb = mref == -INFINITY ? 0.f : mref;
                const float xs_eff = kBias ? 1.f : xscale;   // the bias path holds scaled scores
                // P_b last fed the product of chunk gc-2, which must be done
                if (gc >= 2) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&pempty[b], ((gc >> 1) & 1) ^ 1, abort_flag, p.err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const uint64_t xs2 = f2(xs_eff, xs_eff), nb2 = f2(-mb, -mb);
                uint64_t lc2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};   // partial row sums (two chains)
                // p of each 32-key group, packed, into its 16 columns of P_b;
                // masked scores hold the value that never wins, so p is 0 there
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    uint32_t pk[16];
                    if (gempty[gi]) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pk[e] = 0u;
                    } else {
                        const uint32_t *xg = x + 32 * gi;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float y0, y1;
                            f2split(fma2(f2(__uint_as_float(xg[2 * e]), __uint_as_float(xg[2 * e + 1])), xs2, nb2),
                                    y0, y1);
                            float p0 = ex2(y0), p1 = ex2(y1);
                            lc2[e & 1] = add2(lc2[e & 1], f2(p0, p1));   // the row sum is before dropout
                            if constexpr (kDrop) {   // dropped: 0 (kept: scaled in the epilogue)
                                if (!((keep[gi] >> (2 * e)) & 1u)) p0 = 0.f;
                                if (!((keep[gi] >> (2 * e + 1)) & 1u)) p1 = 0.f;
                            }
                            pk[e] = pack2<T>(p0, p1);
                        }
                    }
                    tmem_st16(lane_base + kColP + 64 * b + 32 * half + 16 * gi, pk);
                }
                float l0, l1;
                f2split(add2(lc2[0], lc2[1]), l0, l1);
                const bool rescale = raise && m != -INFINITY;
                const float corr = rescale ? ex2(m - mref) : 1.f;
                l = l * corr + (l0 + l1);
                const bool resc_any = __any_sync(0xffffffffu, rescale);
                if ((resc_any || epi_pend) && gc >= 1) {
                    // the product of chunk gc-1 (the last one of the previous
                    // tile, in a tile's first chunk) is done: O may be
                    // rescaled or read out
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&pempty[b ^ 1], ((gc - 1) >> 1) & 1, abort_flag, p.err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                // a rescale never happens in a tile's first chunk (m is -inf
                // there), so never together with the epilogue
                if (resc_any) {
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t o[32];
                        tmem_ld32(o_mine + 32 * hh, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st32(o_mine + 32 * hh, o);
                    }
                }
                // the previous tile's O stays in place until this chunk's P is signalled
                if (epi_pend && !epilogue()) {
                    ok = false;
                    break;
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive_warp(&pfull[b]);    // P_b (and the rescaled O) are in tensor memory
                m = mref;
            }
            if (!ok) break;
            // the epilogue of this tile runs in the next tile's first chunk
            epi_pend = true;
            epi_m = m;
            epi_l = l;
            epi_ok = qq < tl.nr;
            epi_row = (long long)tl.bh * g.n + tl.r + (long long)g.s * qq;
            epi_it = it;
            ++it;
        }
        if (ok && epi_pend && gc >= 1) {
            // the last tile's epilogue: its last P.V product read P_{(gc-1) mod 2}
            if (__all_sync(0xffffffffu, mbar_wait(&pempty[(gc - 1) & 1], ((gc - 1) >> 1) & 1, abort_flag, p.err))) {
                tc_fence_after();
                epilogue();
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
    const float *Q = p.Q + dense_row(g, R, g.rs_p);
    const float *K = p.K + dense_row(g, bh * g.n, g.rs_p);   // row j of the slice: j * ks
    const float *V = p.V + dense_row(g, bh * g.n, g.rs_p);
    const long long ks = g.rs_p ? g.rs_p : g.hd;
    const float qc = c < g.hd ? *GP(g.bnd, Q + c) : 0.f;
    const int t_lo = max(0, g.w - i / g.s);
    const int t_hi = min(g.D - 1, g.w + (g.n - 1 - i) / g.s);
    float m = -INFINITY, l = 0.f, acc = 0.f;
    for (int t = t_lo; t <= t_hi; ++t) {
        const long long j = (long long)i + (long long)(t - g.w) * g.s;
        float x = c < g.hd ? qc * *GP(g.bnd, K + j * ks + c) : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) part[wid] = x;
        __syncthreads();
        float sdot = 0.f;
        for (int k = 0; k < nw; ++k) sdot += part[k];
        __syncthreads();
        const float sc = sdot * p.scale +
                         (g.kbias ? *GP(g.bnd, g.kbias + (size_t)(bh / g.h) * g.n + (size_t)j) : 0.f);
        const float m_new = fmaxf(m, sc);
        const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
        const float pv = expf(sc - m_new);
        l = l * corr + pv;   // the row sum is before dropout
        if (c < g.hd) acc = acc * corr + pv * drop_factor(g, bh, i, j) * *GP(g.bnd, V + j * ks + c);
        m = m_new;
    }
    if (c < g.hd) *GP(g.bnd, p.O + dense_row(g, R, g.rs_o) + c) = acc / l;
    if (c == 0 && p.lse) *GP(g.bnd, p.lse + R) = m + logf(l);
}

template <typename T, bool kBias, bool kDrop, bool kGlob = false>
cudaError_t launch_t(const TmapSet &mq, const TmapSet &mk, const TmapSet &mv, const AttnArgs &a,
                     cudaStream_t st, const GlobArgs *gl = nullptr) {
    const long long tiles = (long long)((a.g.nsub + kBQ - 1) / kBQ) * a.g.s * a.g.BH;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const void *fn = reinterpret_cast<const void *>(k_band_attention_fwd<T, kBias, kDrop, kGlob>);
    const size_t smem = kSmemBytes + (kGlob ? (size_t)((a.g.n + 31) / 32) * 4 : 0);
    cudaError_t e = ensure_smem(fn, (int)smem);
    if (e != cudaSuccess) return e;
    // persistent CTAs: as many as fit at once (one per SM), at most one per tile
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long long slots = (long long)sms * per_sm;
    const int grid = (int)(tiles < slots ? tiles : slots);
    GlobArgs none;
    none.G = 0;
    k_band_attention_fwd<T, kBias, kDrop, kGlob><<<grid, kThreads, smem, st>>>(mq, mk, mv, a, gl ? *gl : none);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band_attention_f32(const AttnArgsF32 &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    const int threads = ((a.g.hd + 31) / 32) * 32;
    k_band_attention_f32<<<(unsigned)rows, threads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_band_attention_glob(DType dt, const TmapSet &mapQ, const TmapSet &mapK,
                                       const TmapSet &mapV, const AttnArgs &a, const GlobArgs &gl,
                                       cudaStream_t st) {
    if (a.g.kbias) {   // the key bias of the band keys (global keys: their own kernels)
        if (dt == kF16) return launch_t<__half, true, false, true>(mapQ, mapK, mapV, a, st, &gl);
        return launch_t<__nv_bfloat16, true, false, true>(mapQ, mapK, mapV, a, st, &gl);
    }
    if (dt == kF16) return launch_t<__half, false, false, true>(mapQ, mapK, mapV, a, st, &gl);
    return launch_t<__nv_bfloat16, false, false, true>(mapQ, mapK, mapV, a, st, &gl);
}

cudaError_t launch_band_attention_tc(DType dt, const TmapSet &mapQ, const TmapSet &mapK,
                                     const TmapSet &mapV, const AttnArgs &a, cudaStream_t st) {
    const int v = (a.g.kbias ? 1 : 0) + (a.g.drop_t > 0 ? 2 : 0);
    if (dt == kF16) {
        switch (v) {
            case 0: return launch_t<__half, false, false>(mapQ, mapK, mapV, a, st);
            case 1: return launch_t<__half, true, false>(mapQ, mapK, mapV, a, st);
            case 2: return launch_t<__half, false, true>(mapQ, mapK, mapV, a, st);
            default: return launch_t<__half, true, true>(mapQ, mapK, mapV, a, st);
        }
    }
    switch (v) {
        case 0: return launch_t<__nv_bfloat16, false, false>(mapQ, mapK, mapV, a, st);
        case 1: return launch_t<__nv_bfloat16, true, false>(mapQ, mapK, mapV, a, st);
        case 2: return launch_t<__nv_bfloat16, false, true>(mapQ, mapK, mapV, a, st);
        default: return launch_t<__nv_bfloat16, true, true>(mapQ, mapK, mapV, a, st);
    }
}

}  // namespace swab
