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
// and their barriers carry straight on from one tile into the next (the
// next tile's Q and K/V loads and its first Q.K^T product overlap the
// current tile's epilogue).  For chunk c (128 keys) of a tile:
//   1. MMA warp: S_c = Q . K_c^T (tcgen05, M = 128 queries, N = 128 keys,
//      K = 64) into TMEM score buffer c%2;
//   2. softmax warps: four per TMEM lane quarter, warp part j owning chunk
//      columns [32j, 32j+32) of its 32 rows (thread = query row).  Each keeps
//      its own reference max m (log2 domain) and sum l; m is raised only when
//      the chunk's largest score exceeds it by more than 2^8, so p = 2^(x-m)
//      <= 2^8 stays well inside fp16/bf16.  p is written as the K-major,
//      128-B-swizzled A operand of the next product;
//   3. MMA warp: O_j += P_c[:, part j] . V_c[part j] into part j's own fp32
//      accumulator in TMEM (4 x 64 columns), so no accumulator lives in
//      registers; when a part raises m it rescales its own accumulator rows
//      in place (tcgen05.ld / st) before the product that uses the new m.
// Tile epilogue: the four parts of a row exchange (m_j, l_j) through shared
// memory; part j then reads channels [16j, 16j+16) of all four accumulators,
// combines them (O = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j) and
// writes them out; lse = M ln 2 + ln L.  The chunk sequence runs on across
// tiles: a tile's epilogue runs in the next tile's first chunk, after that
// chunk's softmax and before its P tile is signalled (its P.V product
// overwrites the accumulators), so the next tile's first Q.K^T and softmax
// overlap the tile's last P.V.
//
// Warps: 0 = TMA producer (Q double-buffered, K and V chunks into a 3-stage
// ring), 1 = TMEM owner + MMA issuer, 2..17 = softmax / epilogue.  Every
// wait is a bounded mbarrier wait (no bar.sync inside the loops), so a
// timeout anywhere lets every warp leave.
#include <type_traits>

#include "swab_internal.h"

namespace swab {
namespace {

constexpr int kBQ = 128;        // queries per tile (M)
constexpr int kBK = 128;        // keys per chunk (N of S, K of P.V)
constexpr int kStages = 3;      // K/V ring
constexpr int kParts = 4;       // key parts of a chunk: 32 keys each
constexpr int kWorkerWarps = 4 * kParts;
constexpr int kWorkers = 32 * kWorkerWarps;     // 512
constexpr int kThreads = 64 + kWorkers;         // producer, MMA, softmax warps
constexpr int kQBytes = kBQ * 128;              // 16 KB
constexpr int kKBytes = kBK * 128;              // 16 KB
constexpr int kStageBytes = 2 * kKBytes;        // K and V: 32 KB
constexpr int kPBytes = kBQ * kBK * 2;          // 32 KB (two 64-key K-atoms)
constexpr int kMlBytes = 2 * kParts * kBQ * 8;  // (m, l) exchange, two tile parities
constexpr int kBiasSlotBytes = kWorkerWarps * 32 * 4;  // key bias of each warp's 32 keys
constexpr int kSmemBytes =
    2 * kQBytes + kStages * kStageBytes + 2 * kPBytes + kMlBytes + kBiasSlotBytes + 1024 + 1024;
constexpr uint32_t kTmemCols = 512;             // S: 2 x 128, O: 4 parts x 64
constexpr uint32_t kTmemO = 256;                // O of part j at 256 + 64 j
constexpr float kSlack = 8.f;                   // log2 headroom of the reference max

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Largest (kMin: smallest) of 32 values: four independent 8-value chains.
template <bool kMin>
__device__ __forceinline__ float reduce32(const float (&x)[32]) {
    float c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float *y = x + 8 * k;
        float a = kMin ? min3(y[0], y[1], y[2]) : max3(y[0], y[1], y[2]);
        a = kMin ? min3(a, y[3], y[4]) : max3(a, y[3], y[4]);
        a = kMin ? min3(a, y[5], y[6]) : max3(a, y[5], y[6]);
        c[k] = kMin ? fminf(a, y[7]) : fmaxf(a, y[7]);
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
    // masked), so each softmax warp's 32 keys of a chunk are one dropout block
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
    uint8_t *qtile = base;                               // 2 x 16 KB
    uint8_t *kv = base + 2 * kQBytes;                    // stage st: K at +0, V at +kKBytes
    uint8_t *pbuf = kv + kStages * kStageBytes;          // 2 x 32 KB
    float2 *mlx = reinterpret_cast<float2 *>(pbuf + 2 * kPBytes);  // [2][kParts][kBQ]
    float *bslots = reinterpret_cast<float *>(pbuf + 2 * kPBytes + kMlBytes);  // [16 warps][32]
    uint64_t *bars = reinterpret_cast<uint64_t *>(pbuf + 2 * kPBytes + kMlBytes + kBiasSlotBytes);
    uint64_t *qfull = bars;                  // [2]
    uint64_t *qempty = qfull + 2;            // [2]
    uint64_t *kvfull = qempty + 2;           // [kStages]
    uint64_t *kvempty = kvfull + kStages;    // [kStages]
    uint64_t *sfull = kvempty + kStages;     // [2]
    uint64_t *sempty = sfull + 2;            // [2] count kWorkers
    uint64_t *pfull = sempty + 2;            // [2] count kWorkers
    uint64_t *ofull = pfull + 2;             // 1: P.V product of a chunk done
    uint64_t *mlbar = ofull + 1;             // [4] per lane quarter, count 128
    uint64_t *mmadone = mlbar + 4;           // 1: drain of the MMA pipe at exit
    uint64_t *drain = mmadone + 1;           // 1 int: never set (drain waits ignore aborts)
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(drain);
    // global tokens: bit j of gbits marks position j as global (the band
    // excludes those keys; they are attended through their own columns)
    uint32_t *gbits = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(bars) + 1024);

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
            mbar_init(&sempty[i], kWorkers);
            mbar_init(&pfull[i], kWorkers);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
        }
        mbar_init(ofull, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&mlbar[i], 128);
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

    // The producer and MMA warps run their loops warp-uniformly (every lane
    // walks the tiles and waits on the barriers) and only lane 0 issues the
    // copies, products and commits.
    if (warp == 0) {
        uint32_t gc = 0, it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            Tile tl;
            if (!decode_tile(g, t, xt, tl)) continue;
            const CUtensorMap *mq = &mapQ.m[tl.r], *mk = &mapK.m[tl.r], *mv = &mapV.m[tl.r];
            const int qb = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&qempty[qb], ((it >> 1) & 1) ^ 1, abort_flag, p.err)))
                break;
            if (lane == 0) {
                tma_prefetch_desc(mq);
                tma_prefetch_desc(mk);
                tma_prefetch_desc(mv);
                mbar_arrive_expect_tx(&qfull[qb], kQBytes);
                tma_load_dense(qtile + qb * kQBytes, mq, &qfull[qb], tl.a0, tl.bh, g.h, g.rs_p != 0);
            }
            __syncwarp();
            ++it;
            for (int c = 0; c < tl.nck; ++c) {
                const int st = gc % kStages;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&kvempty[st], ((gc / kStages) & 1) ^ 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&kvfull[st], kStageBytes);
                    uint8_t *stage = kv + st * kStageBytes;
                    tma_load_dense(stage, mk, &kvfull[st], tl.kb_lo + c * kBK, tl.bh, g.h, g.rs_p != 0);
                    tma_load_dense(stage + kKBytes, mv, &kvfull[st], tl.kb_lo + c * kBK, tl.bh, g.h,
                                   g.rs_p != 0);
                }
                __syncwarp();
                ++gc;
            }
        }
        // every copy issued lands before the CTA may exit (the last use of
        // each stage and Q buffer; earlier ones completed before reuse)
        for (uint32_t k = gc > (uint32_t)kStages ? gc - kStages : 0; k < gc; ++k)
            mbar_wait(&kvfull[k % kStages], (k / kStages) & 1, no_abort, nullptr, 100000000ull);
        for (uint32_t k = it > 2u ? it - 2 : 0; k < it; ++k)
            mbar_wait(&qfull[k & 1], (k >> 1) & 1, no_abort, nullptr, 100000000ull);
    } else if (warp == 1) {
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        constexpr uint32_t idesc_s = idesc_f16(kBQ, kBK, kBf16, false, false);
        constexpr uint32_t idesc_o = idesc_f16(kBQ, 64, kBf16, false, true);
        // Shared-memory descriptors are built once; a buffer, stage or K step
        // only moves the start address field (address >> 4, which stays below
        // 2^14 for any shared-memory address), so each one is a 64-bit add of
        // a compile-time offset.
        const uint64_t qdesc = sdesc_sw128(smem_u32(qtile), 16, 1024);
        const uint64_t kdesc = sdesc_sw128(smem_u32(kv), 16, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(kv + kKBytes), 1024, 1024);
        const uint64_t pdesc = sdesc_sw128(smem_u32(pbuf), 16, 1024);
        // O_j (+)= P[:, part j] . V[part j]: the P.V product of chunk gg
        auto issue_pv = [&](uint32_t gg, bool first) -> bool {
            const int st = gg % kStages;
            const int b = gg & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&pfull[b], (gg >> 1) & 1, abort_flag, p.err)))
                return false;
            tc_fence_after();
            const uint64_t pa = pdesc + (uint64_t)((b * kPBytes) >> 4);
            const uint64_t va = vdesc + (uint64_t)((st * kStageBytes) >> 4);
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < kParts; ++j) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        // keys 32j + 16kk ..: atom j/2 of P, rows 32j + 16kk.. of V
                        mma_f16_ss(tmem + kTmemO + 64 * j,
                                   pa + (((j >> 1) * (kPBytes / 2) + (j & 1) * 64 + kk * 32) >> 4),
                                   va + (((2 * j + kk) * 2048) >> 4), idesc_o,
                                   (first && kk == 0) ? 0u : 1u);
                    }
                }
                mma_commit(ofull);
                mma_commit(&kvempty[st]);
            }
            __syncwarp();
            return true;
        };
        uint32_t gc = 0, it = 0, prev = 0;
        bool ok = true, have_prev = false, prev_first = false;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            Tile tl;
            if (!decode_tile(g, t, xt, tl)) continue;
            const int qb = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&qfull[qb], (it >> 1) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            const uint64_t qa = qdesc + (uint64_t)((qb * kQBytes) >> 4);
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int st = gc % kStages;
                const int b = gc & 1;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&kvfull[st], (gc / kStages) & 1, abort_flag, p.err) &&
                                    mbar_wait(&sempty[b], ((gc >> 1) & 1) ^ 1, abort_flag, p.err));
                if (!ok) break;
                tc_fence_after();
                const uint64_t ka = kdesc + (uint64_t)((st * kStageBytes) >> 4);
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ss(tmem + b * kBK, qa + 2 * k, ka + 2 * k, idesc_s, k > 0);
                    if (c == tl.nck - 1) mma_commit(&qempty[qb]);
                    mma_commit(&sfull[b]);
                }
                __syncwarp();
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
        if (lane == 0) mma_commit(mmadone);
        __syncwarp();
        mbar_wait(mmadone, 0, no_abort, nullptr, 100000000ull);
    } else {
        // ---------------- softmax warps: thread = query row ----------------
        const int quarter = warp & 3;
        const int part = (warp - 2) >> 2;
        const int q = quarter * 32 + lane;
        const float xscale = p.scale * 1.4426950408889634f;
        const bool neg_scale = xscale < 0.f;
        const float dscale = 256.f / (256.f - (float)g.drop_t);   // kept values' scale
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        const uint32_t o_mine = lane_base + kTmemO + 64 * part;
        uint32_t gc = 0, it = 0;
        bool ok = true;
        bool epi_pend = false, epi_ok = false;
        float epi_m = 0.f, epi_l = 0.f;
        long long epi_row = 0;
        uint32_t epi_it = 0;
        // the epilogue of tile epi_it (row epi_row, this part's (epi_m, epi_l));
        // the caller has waited for the tile's last P.V product
        auto epilogue = [&]() -> bool {
            epi_pend = false;
            float2 *ml = mlx + (epi_it & 1) * kParts * kBQ;
            ml[part * kBQ + q] = make_float2(epi_m, epi_l);
            mbar_arrive(&mlbar[quarter]);
            if (!__all_sync(0xffffffffu, mbar_wait(&mlbar[quarter], epi_it & 1, abort_flag, p.err)))
                return false;
            float M = -INFINITY;
            float2 e[kParts];
#pragma unroll
            for (int j = 0; j < kParts; ++j) {
                e[j] = ml[j * kBQ + q];
                M = fmaxf(M, e[j].x);
            }
            float f[kParts], L = 0.f;
#pragma unroll
            for (int j = 0; j < kParts; ++j) {
                f[j] = e[j].x == -INFINITY ? 0.f : ex2(e[j].x - M);
                L += e[j].y * f[j];
            }
            const float inv = (kDrop ? dscale : 1.f) / L;   // kept values scaled once, here
            // channels [16 part, 16 part + 16) of the four accumulators, two at a time
            float y[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) y[i] = 0.f;
#pragma unroll
            for (int j0 = 0; j0 < kParts; j0 += 2) {
                uint32_t o0[16], o1[16];
                tmem_ld16(lane_base + kTmemO + 64 * j0 + 16 * part, o0);
                tmem_ld16(lane_base + kTmemO + 64 * (j0 + 1) + 16 * part, o1);
                tmem_ld_wait();
                const float f0 = f[j0] * inv, f1 = f[j0 + 1] * inv;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    y[i] = fmaf(__uint_as_float(o1[i]), f1, fmaf(__uint_as_float(o0[i]), f0, y[i]));
            }
            tc_fence_before();   // O may be overwritten once this warp's next P tile is signalled
            if (epi_ok) {
                const long long row = epi_row;
                uint4 *o4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.O) + dense_row(g, row, g.rs_o) +
                                                      16 * part);
                o4[0] = make_uint4(pack2<T>(y[0], y[1]), pack2<T>(y[2], y[3]), pack2<T>(y[4], y[5]),
                                   pack2<T>(y[6], y[7]));
                o4[1] = make_uint4(pack2<T>(y[8], y[9]), pack2<T>(y[10], y[11]),
                                   pack2<T>(y[12], y[13]), pack2<T>(y[14], y[15]));
                if (p.lse && part == 0) p.lse[row] = M * 0.6931471805599453f + logf(L);
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
                const int kbase = tl.kb_lo + c * kBK + 32 * part;
                // this row's band inside the part: columns [max(jlo,0), min(jhi,31)]
                const int jlo = max(qq - g.w - kbase, 0);
                const int jhi = min(min(qq + g.wu, tl.kb_hi) - kbase, 31);
                uint32_t vmask = jlo > jhi ? 0u : ((2u << jhi) - 1u) & (0xffffffffu << jlo);
                if constexpr (kGlob) {
                    // column `lane` of the part is key kbase + lane of the residue
                    const int sub = kbase + lane;
                    const int key = tl.r + g.s * sub;
                    const bool isg = sub < tl.nr && ((gbits[key >> 5] >> (key & 31)) & 1u);
                    vmask &= ~__ballot_sync(0xffffffffu, isg);
                }
                const bool full = __all_sync(0xffffffffu, vmask == 0xffffffffu);
                const bool empty = __all_sync(0xffffffffu, vmask == 0u);
                // dropout keep bits of this row's 32 keys (one Philox block:
                // kbase is a multiple of 32)
                uint32_t keep = 0xffffffffu;
                if constexpr (kDrop) {
                    if (!empty && qq < tl.nr) {
                        unsigned long long wv[4];
                        philox4x64_10((unsigned long long)(kbase / 32),
                                      (unsigned long long)(tl.r + (long long)g.s * qq),
                                      (unsigned long long)tl.bh, 0, g.seed, 0, wv);
                        keep = keep_bits32(wv, g.drop_t);
                    }
                }
                float kb = 0.f;   // key bias (log2 units) of this part's key `lane`
                if constexpr (kBias) {
                    if (!empty && kbase + lane < tl.nr)
                        kb = __ldg(g.kbias + (size_t)(tl.bh / g.h) * g.n + tl.r + (size_t)g.s * (kbase + lane)) *
                             1.4426950408889634f;
                }
                bool w_ok = mbar_wait(&sfull[b], (gc >> 1) & 1, abort_flag, p.err);
                if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
                tc_fence_after();
                float x[32];
                {
                    uint32_t v[32];
                    tmem_ld32(lane_base + b * kBK + 32 * part, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
                }
                tc_fence_before();
                mbar_arrive(&sempty[b]);   // the scores are in registers
                // P tile b last fed the product of chunk gc-2, which is done
                const uint32_t prow = smem_u32(pbuf + b * kPBytes) + (part >> 1) * (kPBytes / 2) + q * 128;
                float cmax = -INFINITY, lc = 0.f;
                if (empty) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int piece = (part & 1) * 4 + u;
                        sts16(prow + ((piece ^ (q & 7)) << 4), make_uint4(0u, 0u, 0u, 0u));
                    }
                } else {
                    if constexpr (kBias) {
                        // scaled score plus the key bias, in log2 units: the
                        // scale is folded in here, so the passes below see
                        // scale 1
                        float *slot = bslots + (warp - 2) * 32;
                        slot[lane] = kb;
                        __syncwarp();
                        const float4 *b4 = reinterpret_cast<const float4 *>(slot);
                        const uint64_t xs2 = f2(xscale, xscale);
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const float4 bb = b4[u];
                            f2split(fma2(f2(x[4 * u], x[4 * u + 1]), xs2, f2(bb.x, bb.y)), x[4 * u], x[4 * u + 1]);
                            f2split(fma2(f2(x[4 * u + 2], x[4 * u + 3]), xs2, f2(bb.z, bb.w)), x[4 * u + 2],
                                    x[4 * u + 3]);
                        }
                        __syncwarp();
                    }
                    // chunk max of the scaled scores from the raw ones: the
                    // largest raw score for a positive scale, the smallest
                    // for a negative one; columns outside the band are
                    // replaced by the value that never wins
                    const bool neg = kBias ? false : neg_scale;
                    if (!full) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (!((vmask >> i) & 1u)) x[i] = neg ? INFINITY : -INFINITY;
                    }
                    const float vm = neg ? reduce32<true>(x) : reduce32<false>(x);
                    cmax = vmask == 0u ? -INFINITY : vm * (kBias ? 1.f : xscale);
                }
                const bool raise = m == -INFINITY || cmax > m + kSlack;
                const float mref = raise ? cmax : m;
                if (!empty) {
                    const float mb = mref == -INFINITY ? 0.f : mref;
                    const float xs_eff = kBias ? 1.f : xscale;   // the bias path holds scaled scores
                    const uint64_t xs2 = f2(xs_eff, xs_eff), nb2 = f2(-mb, -mb);
                    uint64_t lc2 = f2(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 8 * u + 2 * e;
                            float y0, y1;
                            f2split(fma2(f2(x[i], x[i + 1]), xs2, nb2), y0, y1);
                            float p0 = ex2(y0), p1 = ex2(y1);
                            if (!full) {
                                if (!((vmask >> i) & 1u)) p0 = 0.f;
                                if (!((vmask >> (i + 1)) & 1u)) p1 = 0.f;
                            }
                            lc2 = add2(lc2, f2(p0, p1));   // the row sum is before dropout
                            if constexpr (kDrop) {   // dropped: 0 (kept: scaled in the epilogue)
                                if (!((keep >> i) & 1u)) p0 = 0.f;
                                if (!((keep >> (i + 1)) & 1u)) p1 = 0.f;
                            }
                            pk[e] = pack2<T>(p0, p1);
                        }
                        const int piece = (part & 1) * 4 + u;
                        sts16(prow + ((piece ^ (q & 7)) << 4), make_uint4(pk[0], pk[1], pk[2], pk[3]));
                    }
                    float l0, l1;
                    f2split(lc2, l0, l1);
                    lc = l0 + l1;
                }
                const bool rescale = raise && m != -INFINITY;
                const float corr = rescale ? ex2(m - mref) : 1.f;
                l = l * corr + lc;
                if (c > 0 || epi_pend) {
                    // the product of chunk gc-1 has landed in O: it may be
                    // rescaled, or (first chunk of a tile) the previous tile's
                    // accumulators are final
                    w_ok = mbar_wait(ofull, (gc - 1) & 1, abort_flag, p.err);
                    if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
                }
                if (epi_pend) {
                    tc_fence_after();
                    if (!epilogue()) { ok = false; break; }
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    tc_fence_after();
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        uint32_t o[32];
                        tmem_ld32(o_mine + 32 * h, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st32(o_mine + 32 * h, o);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                fence_proxy_async_smem();
                mbar_arrive(&pfull[b]);    // P tile b (and the rescaled O) are ready
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
        if (ok && epi_pend) {
            // the last tile's epilogue: its last P.V product is phase gc-1 of ofull
            if (__all_sync(0xffffffffu, mbar_wait(ofull, (gc - 1) & 1, abort_flag, p.err))) {
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
    const float qc = c < g.hd ? Q[c] : 0.f;
    const int t_lo = max(0, g.w - i / g.s);
    const int t_hi = min(g.D - 1, g.w + (g.n - 1 - i) / g.s);
    float m = -INFINITY, l = 0.f, acc = 0.f;
    for (int t = t_lo; t <= t_hi; ++t) {
        const long long j = (long long)i + (long long)(t - g.w) * g.s;
        float x = c < g.hd ? qc * K[j * ks + c] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) part[wid] = x;
        __syncthreads();
        float sdot = 0.f;
        for (int k = 0; k < nw; ++k) sdot += part[k];
        __syncthreads();
        const float sc = sdot * p.scale +
                         (g.kbias ? g.kbias[(size_t)(bh / g.h) * g.n + (size_t)j] : 0.f);
        const float m_new = fmaxf(m, sc);
        const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
        const float pv = expf(sc - m_new);
        l = l * corr + pv;   // the row sum is before dropout
        if (c < g.hd) acc = acc * corr + pv * drop_factor(g, bh, i, j) * V[j * ks + c];
        m = m_new;
    }
    if (c < g.hd) p.O[dense_row(g, R, g.rs_o) + c] = acc / l;
    if (c == 0 && p.lse) p.lse[R] = m + logf(l);
}

template <typename T, bool kBias, bool kDrop, bool kGlob = false>
cudaError_t launch_t(const TmapSet &mq, const TmapSet &mk, const TmapSet &mv, const AttnArgs &a,
                     cudaStream_t st, const GlobArgs *gl = nullptr) {
    const long long tiles = (long long)((a.g.nsub + kBQ - 1) / kBQ) * a.g.s * a.g.BH;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = (int)(tiles < sms ? tiles : sms);
    const size_t smem = kSmemBytes + (kGlob ? (size_t)((a.g.n + 31) / 32) * 4 : 0);
    cudaError_t e =
        ensure_smem(reinterpret_cast<const void *>(k_band_attention_fwd<T, kBias, kDrop, kGlob>), smem);
    if (e != cudaSuccess) return e;
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
