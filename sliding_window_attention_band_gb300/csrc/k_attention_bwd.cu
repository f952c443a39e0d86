// k_attention_bwd.cu -- fused backward of sliding-window attention: dQ, dK,
// dV of O = softmax_band(scale * Q K^T) V without materialising any band
// tensor.  The banded products are those of "Developing a faster schedule
// for Longformer's kernel" (TVM forum, post 6: the forward product and the two
// backward products); the softmax derivative is the textbook one:
//     P  = exp(scale * Q K^T - lse)         (lse from the forward)
//     dP = dO V^T,   delta_i = dO_i . O_i,   dS = P * (dP - delta)
//     dQ = scale * dS K,   dK = scale * dS^T Q,   dV = P^T dO
// all restricted to the band (and to keys inside the sequence).
//
// Deterministic, no atomics: three kernels.
//   k_bwd_delta     delta_i = dO_i . O_i into a caller-provided fp32 workspace.
//   k_bwd_dkdv      one CTA per 128 KEYS of one residue; walks the queries
//                   whose band contains them, 128 at a time:
//                   S^T = K Q_c^T and dP^T = V dO_c^T (tcgen05, TMEM lane =
//                   key), P^T and dS^T computed per key row and written as
//                   K-major A operands, then dV += P^T dO_c and
//                   dK += dS^T Q_c accumulate in TMEM.
//   k_bwd_dq        one CTA per 128 QUERIES (the fused forward's layout):
//                   S = Q K_c^T and dP = dO V_c^T, dS per query row, then
//                   dQ += dS K_c in TMEM.
// The dense tiles staged by TMA serve twice: K-major as the K=64 operand of
// the score products and MN-major (rows along K) as the B operand of the
// gradient products.
#include <mutex>
#include <type_traits>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 2;   // site id of the bounds checks

namespace swab {

// Device scratch for band_attention_bwd_noalloc: the per-row delta that the
// regular entry point keeps in a caller-provided workspace.  It is a
// module-scope array, so every GPU that loads the library holds it (16 MiB)
// until the process exits, and every call of that entry point on a device
// shares it.
static __device__ __align__(256) float g_noalloc_delta[SWAB_NOALLOC_MAX_ROWS];

// Device address of g_noalloc_delta on the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up
// with cudaGetSymbolAddress, once per device (the first call on a device does
// it) and cached.  The lookup may load the module, which must not happen
// while `st` is being captured: a first call under capture is refused
// (cudaErrorStreamCaptureUnsupported) before anything is looked up.
cudaError_t noalloc_delta_scratch(float **out, cudaStream_t st) {
    static std::mutex mu;
    static float *cache[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(st, &cs);
        if (e != cudaSuccess) return e;
        if (cs != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_delta);
        if (e != cudaSuccess) return e;
        cache[dev] = static_cast<float *>(ptr);
    }
    *out = cache[dev];
    return cudaSuccess;
}

namespace {

constexpr int kB = 128;           // rows per CTA and per chunk
constexpr int kThreads = 320;     // producer, MMA, 8 worker warps (2 per TMEM lane quarter)
constexpr int kWorkers = 256;
constexpr int kTile = kB * 128;   // 16 KB: 128 rows x 64 halves
constexpr int kStages = 2;
constexpr int kOpBytes = kB * kB * 2;  // 32 KB: a 128 x 128 16-bit A operand (two K-atoms)
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Write 32 packed values (16 words) of row `row` into a K-major 128-B-swizzled
// 128 x 128 operand at key/query group `grp` (32 columns).
__device__ __forceinline__ void store_op_row(uint32_t op_addr, int row, int grp,
                                             const uint32_t (&pk)[16]) {
    const uint32_t atom = op_addr + (grp >> 1) * (kOpBytes / 2) + row * 128;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int piece = (grp & 1) * 4 + u;
        sts16(atom + ((piece ^ (row & 7)) << 4),
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
    }
}

// D (+)= A[128 x 128, K-major smem operand] * B[K = 128 rows of 64, MN-major]
__device__ __forceinline__ void mma_op_by_rows(uint32_t d, uint32_t a_addr, uint32_t b_addr,
                                               uint32_t idesc, bool accumulate_first) {
#pragma unroll
    for (int k = 0; k < kB / 16; ++k) {
        const uint32_t a = a_addr + (k >> 2) * (kOpBytes / 2) + (k & 3) * 32;
        mma_f16_ss(d, sdesc_sw128(a, 16, 1024), sdesc_sw128(b_addr + 2048 * k, 1024, 1024), idesc,
                   (accumulate_first || k > 0) ? 1u : 0u);
    }
}

// D = A[128 x 64, K-major tile] * B[128 x 64, K-major tile]^T
__device__ __forceinline__ void mma_tiles(uint32_t d, uint32_t a_addr, uint32_t b_addr,
                                          uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_f16_ss(d, sdesc_sw128(a_addr + 32 * k, 16, 1024), sdesc_sw128(b_addr + 32 * k, 16, 1024),
                   idesc, k > 0);
}

// Programmatic dependent launch: a kernel launched with the stream
// serialization attribute may start while the kernel before it runs; it
// waits for that kernel's completion (and its memory) before reading what it
// wrote.  Without the attribute both instructions do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------------------
// delta_i = dO_i . O_i: 8 lanes per row, 16-byte loads, each warp keeps 4
// groups of 4 rows (16 rows, 8 loads per lane) in flight before reducing.
// ---------------------------------------------------------------------------
constexpr int kDeltaRowsPerWarp = 16;

template <typename T>
__global__ void __launch_bounds__(256) k_bwd_delta(const BwdArgs p) {
    pdl_trigger();   // the one-pass kernel may start its loads
    const long long rows = (long long)p.g.BH * p.g.n;
    const int lane = threadIdx.x & 31;
    const long long warp_row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kDeltaRowsPerWarp;
    const uint4 *O = reinterpret_cast<const uint4 *>(p.O);
    const uint4 *dO = reinterpret_cast<const uint4 *>(p.dO);
    uint4 o[kDeltaRowsPerWarp / 4], d[kDeltaRowsPerWarp / 4];
#pragma unroll
    for (int k = 0; k < kDeltaRowsPerWarp / 4; ++k) {
        const long long R = warp_row0 + 4 * k + (lane >> 3);
        if (R < rows) {
            const long long off = dense_row(p.g, R, p.g.rs_o) / 8;   // 8 elements per 16 bytes
            o[k] = ldg16(GP(p.g.bnd, O + off + (lane & 7)));
            d[k] = ldg16(GP(p.g.bnd, dO + off + (lane & 7)));
        } else {
            o[k] = d[k] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int k = 0; k < kDeltaRowsPerWarp / 4; ++k) {
        const uint32_t ow[4] = {o[k].x, o[k].y, o[k].z, o[k].w};
        const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
        float v = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v = fmaf(lo16<T>(ow[u]), lo16<T>(dw[u]), fmaf(hi16<T>(ow[u]), hi16<T>(dw[u]), v));
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        const long long R = warp_row0 + 4 * k + (lane >> 3);
        if ((lane & 7) == 0 && R < rows) *GP(p.g.bnd, p.delta + R) = v;
    }
    if (p.dqacc) {
        // the one-pass backward adds dQ contributions into an fp32 accumulator:
        // clear this warp's rows of it (16 rows x 64 floats)
        float4 *acc = reinterpret_cast<float4 *>(p.dqacc);
#pragma unroll
        for (int k = 0; k < kDeltaRowsPerWarp * 16 / 32; ++k) {
            const int idx = k * 32 + lane;
            const long long R = warp_row0 + idx / 16;
            if (R < rows) *GP(p.g.bnd, acc + R * 16 + (idx & 15)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// dQ = scale * accumulator, rounded to the output type: 8 channels per thread.
// The accumulator is dead once read (the next call clears it again), so its
// 128-byte lines are then dropped from L2 without being written back: the
// clearing and the reduce-adds never cost DRAM writes.
template <typename T>
__global__ void __launch_bounds__(256) k_bwd_dq_out(const BwdArgs p) {
    pdl_wait();   // every dQ addition of the one-pass kernel has landed
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // 8-channel group
    const long long groups = (long long)p.g.BH * p.g.n * 8;
    if (i < groups) {
        const float4 *acc = reinterpret_cast<const float4 *>(p.dqacc) + 2 * i;
        const float4 a = *GP(p.g.bnd, acc), b = *GP(p.g.bnd, acc + 1);
        const float c = p.scale;
        const long long off = dense_row(p.g, i >> 3, p.g.rs_p) / 8 + (i & 7);   // row i / 8, group i % 8
        *GP(p.g.bnd, reinterpret_cast<uint4 *>(p.dQ) + off) = make_uint4(pack2<T>(c * a.x, c * a.y), pack2<T>(c * a.z, c * a.w),
                                                        pack2<T>(c * b.x, c * b.y), pack2<T>(c * b.z, c * b.w));
    }
    // four consecutive threads read one 128-byte line (rows are 256 bytes);
    // their loads are complete (the values were used above) when the warp
    // synchronises, and the first of the four drops the line
    __syncwarp();
    if ((reinterpret_cast<uintptr_t>(p.dqacc) & 127u) == 0 && (i & 3) == 0 && i < groups)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(GPN(p.g.bnd, reinterpret_cast<const float4 *>(p.dqacc) + 2 * i, 128))
                     : "memory");
}

// ---------------------------------------------------------------------------
// dK, dV: one CTA per 128 keys
// ---------------------------------------------------------------------------
constexpr int kSmemDKDV = 2 * kTile + kStages * 2 * kTile + 2 * kOpBytes + 2 * 2 * kB * 4 + 1024 + 1024;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_dkdv(const __grid_constant__ TmapSet mapQ, const __grid_constant__ TmapSet mapK,
               const __grid_constant__ TmapSet mapV, const __grid_constant__ TmapSet mapdO,
               const BwdArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ktile = base;
    uint8_t *vtile = base + kTile;
    uint8_t *stages = base + 2 * kTile;                   // stage: Q chunk, dO chunk
    uint8_t *pt_op = stages + kStages * 2 * kTile;        // P^T  [128 keys x 128 queries]
    uint8_t *dst_op = pt_op + kOpBytes;                   // dS^T
    float *qstat = reinterpret_cast<float *>(dst_op + kOpBytes);  // [2][2][128]: lse*log2e, delta
    uint64_t *bars = reinterpret_cast<uint64_t *>(qstat + 2 * 2 * kB);
    uint64_t *kvfull = bars;                  // 1
    uint64_t *qfull = bars + 1;               // [kStages]
    uint64_t *qempty = qfull + kStages;       // [kStages]
    uint64_t *sfull = qempty + kStages;       // 1
    uint64_t *sempty = sfull + 1;             // 1, count 128
    uint64_t *opfull = sempty + 1;            // 1, count 128
    uint64_t *opempty = opfull + 1;           // 1
    uint64_t *accfull = opempty + 1;          // 1
    uint64_t *statbar = accfull + 1;          // 1, count kWorkers: a chunk's lse, delta written
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(statbar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, bh = blockIdx.z;
    const int nr = residue_len(g.n, g.s, r);
    const int a0 = blockIdx.x * kB;  // first key (sub-index)
    if (a0 >= nr) return;
    const int qb_lo = max(a0 - g.wu, 0);
    const int qb_hi = min(a0 + kB - 1 + g.w, nr - 1);
    const int nck = (qb_hi - qb_lo + kB) / kB;

    if (threadIdx.x == 0) {
        mbar_init(kvfull, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        mbar_init(sfull, 1);
        mbar_init(sempty, kWorkers);
        mbar_init(opfull, kWorkers);
        mbar_init(opempty, 1);
        mbar_init(accfull, 1);
        mbar_init(statbar, kWorkers);
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
    constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap *mq = &mapQ.m[r], *mk = &mapK.m[r], *mv = &mapV.m[r],
                              *mo = &mapdO.m[r];
            mbar_arrive_expect_tx(kvfull, 2 * kTile);
            tma_load_3d(ktile, mk, kvfull, 0, a0, bh);
            tma_load_3d(vtile, mv, kvfull, 0, a0, bh);
            for (int c = 0; c < nck; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                if (!mbar_wait(&qempty[st], ph ^ 1, abort_flag, p.err)) break;
                mbar_arrive_expect_tx(&qfull[st], 2 * kTile);
                uint8_t *sq = stages + st * 2 * kTile;
                tma_load_3d(sq, mq, &qfull[st], 0, qb_lo + c * kB, bh);
                tma_load_3d(sq + kTile, mo, &qfull[st], 0, qb_lo + c * kB, bh);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t id_s = idesc_f16(kB, kB, kBf16, false, false);  // 128x128, both K-major
            const uint32_t id_g = idesc_f16(kB, 64, kBf16, false, true);   // 128x64, B MN-major
            const uint32_t k_addr = smem_u32(ktile), v_addr = smem_u32(vtile);
            bool ok = mbar_wait(kvfull, 0, abort_flag, p.err);
            auto issue_grad = [&](int c) -> bool {
                const int st = c % kStages;
                const uint32_t ph = c & 1;
                if (!mbar_wait(opfull, ph, abort_flag, p.err)) return false;
                tc_fence_after();
                const uint32_t q_addr = smem_u32(stages + st * 2 * kTile);
                const uint32_t o_addr = q_addr + kTile;
                mma_op_by_rows(tmem + kColDV, smem_u32(pt_op), o_addr, id_g, c > 0);
                mma_op_by_rows(tmem + kColDK, smem_u32(dst_op), q_addr, id_g, c > 0);
                mma_commit(opempty);
                mma_commit(&qempty[st]);
                return true;
            };
            for (int c = 0; c < nck && ok; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                ok = mbar_wait(&qfull[st], ph, abort_flag, p.err) &&
                     mbar_wait(sempty, (c & 1) ^ 1, abort_flag, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t q_addr = smem_u32(stages + st * 2 * kTile);
                mma_tiles(tmem + kColS, k_addr, q_addr, id_s);            // S^T  = K Q_c^T
                mma_tiles(tmem + kColDP, v_addr, q_addr + kTile, id_s);   // dP^T = V dO_c^T
                mma_commit(sfull);
                if (c > 0) ok = issue_grad(c - 1);
            }
            if (ok && issue_grad(nck - 1)) mma_commit(accfull);
        }
    } else {
        // ---------------- workers: thread = key row ----------------
        // two warps per TMEM lane quarter; warp half h owns query columns
        // [64h, 64h + 64) of every chunk
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int m = quarter * 32 + lane;
        const int tid = threadIdx.x - 64;  // 0..255
        const int kk = a0 + m;             // key sub-index
        const float xscale = p.scale * kLog2e;
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        bool ok = true;
        for (int c = 0; c < nck; ++c) {
            const int qbase = qb_lo + c * kB;
            // per-query statistics of this chunk into shared memory
            float *ql = qstat + (c & 1) * 2 * kB;
            {
                const int qi = tid & (kB - 1);
                const int qq = qbase + qi;
                const long long row = (long long)bh * g.n + r + (long long)g.s * qq;
                if (tid < kB) ql[qi] = qq < nr ? *GP(g.bnd, p.lse + row) * kLog2e : INFINITY;
                else ql[kB + qi] = qq < nr ? *GP(g.bnd, p.delta + row) : 0.f;
            }
            // every worker's statistics are in (a bounded wait: a timeout
            // anywhere lets every warp leave)
            mbar_arrive(statbar);
            if (!__all_sync(0xffffffffu, mbar_wait(statbar, c & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            // this key's queries inside the chunk: columns [jlo, jhi]
            const int jlo = max(kk - g.wu - qbase, 0);
            const int jhi = min(min(kk + g.w, qb_hi) - qbase, kB - 1);
            const bool key_ok = kk < nr;
            const bool full = __all_sync(0xffffffffu, key_ok && jlo <= 64 * half && jhi >= 64 * half + 63);
            bool w_ok = mbar_wait(sfull, c & 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
            tc_fence_after();
            w_ok = mbar_wait(opempty, (c & 1) ^ 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
            const uint32_t pt = smem_u32(pt_op), dst = smem_u32(dst_op);
            const float4 *ql4 = reinterpret_cast<const float4 *>(ql);
#pragma unroll 1
            for (int grp = 2 * half; grp < 2 * half + 2; ++grp) {
                uint32_t sv[32], dv[32];
                tmem_ld32(lane_base + kColS + grp * 32, sv);
                tmem_ld32(lane_base + kColDP + grp * 32, dv);
                tmem_ld_wait();
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4) {
                    const float4 l4 = ql4[grp * 8 + i4];        // lse*log2e of 4 queries
                    const float4 d4 = ql4[(kB + grp * 32) / 4 + i4];  // delta of the same
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                    const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
                    float pr[4], ds[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int e = 4 * i4 + h;
                        float y = fmaf(__uint_as_float(sv[e]), xscale, -lv[h]);
                        if (!full) {
                            const int j = grp * 32 + e;
                            if (!key_ok || j < jlo || j > jhi) y = -INFINITY;
                        }
                        pr[h] = ex2(y);
                        ds[h] = pr[h] * (__uint_as_float(dv[e]) - dl[h]);
                    }
                    pk[2 * i4] = pack2<T>(pr[0], pr[1]);
                    pk[2 * i4 + 1] = pack2<T>(pr[2], pr[3]);
                    dk[2 * i4] = pack2<T>(ds[0], ds[1]);
                    dk[2 * i4 + 1] = pack2<T>(ds[2], ds[3]);
                }
                store_op_row(pt, m, grp, pk);
                store_op_row(dst, m, grp, dk);
            }
            tc_fence_before();
            mbar_arrive(sempty);
            fence_proxy_async_smem();
            mbar_arrive(opfull);
        }
        const bool acc_ok = ok && mbar_wait(accfull, 0, abort_flag, p.err);
        if (__all_sync(0xffffffffu, acc_ok)) {
            tc_fence_after();
            const bool key_ok = kk < nr;
            const long long row = (long long)bh * g.n + r + (long long)g.s * kk;
            {
                const int which = half;  // half 0 writes dV, half 1 writes dK
                const float mul = which ? p.scale : 1.f;
                T *dst_row = reinterpret_cast<T *>(which ? p.dK : p.dV) + row * 64;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + (which ? kColDK : kColDV) + h * 32, v);
                    tmem_ld_wait();
                    if (key_ok) {
                        uint4 *o4 = reinterpret_cast<uint4 *>(dst_row + h * 32);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            *GP(g.bnd, o4 + u) = make_uint4(
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
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// dQ: one CTA per 128 queries
// ---------------------------------------------------------------------------
constexpr int kSmemDQ = 2 * kTile + kStages * 2 * kTile + 2 * kOpBytes + 1024 + 1024;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_dq(const __grid_constant__ TmapSet mapQ, const __grid_constant__ TmapSet mapK,
             const __grid_constant__ TmapSet mapV, const __grid_constant__ TmapSet mapdO,
             const BwdArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qtile = base;
    uint8_t *otile = base + kTile;                        // dO
    uint8_t *stages = base + 2 * kTile;                   // stage: K chunk, V chunk
    uint8_t *ds_op = stages + kStages * 2 * kTile;        // 2 x [128 queries x 128 keys]
    uint64_t *bars = reinterpret_cast<uint64_t *>(ds_op + 2 * kOpBytes);
    uint64_t *qfull = bars;                   // 1
    uint64_t *kvfull = bars + 1;              // [kStages]
    uint64_t *kvempty = kvfull + kStages;     // [kStages]
    uint64_t *sfull = kvempty + kStages;      // 1
    uint64_t *sempty = sfull + 1;             // 1, count 128
    uint64_t *dsfull = sempty + 1;            // [2], count 128
    uint64_t *dsempty = dsfull + 2;           // [2]
    uint64_t *accfull = dsempty + 2;          // 1
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(accfull + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, bh = blockIdx.z;
    const int nr = residue_len(g.n, g.s, r);
    const int a0 = blockIdx.x * kB;  // first query (sub-index)
    if (a0 >= nr) return;
    const int kb_lo = max(a0 - g.w, 0);
    const int kb_hi = min(a0 + kB - 1 + g.wu, nr - 1);
    const int nck = (kb_hi - kb_lo + kB) / kB;

    if (threadIdx.x == 0) {
        mbar_init(qfull, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
        }
        mbar_init(sfull, 1);
        mbar_init(sempty, kWorkers);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&dsfull[i], kWorkers);
            mbar_init(&dsempty[i], 1);
        }
        mbar_init(accfull, 1);
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
    constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap *mq = &mapQ.m[r], *mk = &mapK.m[r], *mv = &mapV.m[r],
                              *mo = &mapdO.m[r];
            mbar_arrive_expect_tx(qfull, 2 * kTile);
            tma_load_3d(qtile, mq, qfull, 0, a0, bh);
            tma_load_3d(otile, mo, qfull, 0, a0, bh);
            for (int c = 0; c < nck; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                if (!mbar_wait(&kvempty[st], ph ^ 1, abort_flag, p.err)) break;
                mbar_arrive_expect_tx(&kvfull[st], 2 * kTile);
                uint8_t *sk = stages + st * 2 * kTile;
                tma_load_3d(sk, mk, &kvfull[st], 0, kb_lo + c * kB, bh);
                tma_load_3d(sk + kTile, mv, &kvfull[st], 0, kb_lo + c * kB, bh);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t id_s = idesc_f16(kB, kB, kBf16, false, false);
            const uint32_t id_g = idesc_f16(kB, 64, kBf16, false, true);
            const uint32_t q_addr = smem_u32(qtile), o_addr = smem_u32(otile);
            bool ok = mbar_wait(qfull, 0, abort_flag, p.err);
            auto issue_dq = [&](int c) -> bool {
                const int st = c % kStages;
                const int b = c & 1;
                const uint32_t bph = (c >> 1) & 1;
                if (!mbar_wait(&dsfull[b], bph, abort_flag, p.err)) return false;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(stages + st * 2 * kTile);
                mma_op_by_rows(tmem + kColDQ, smem_u32(ds_op + b * kOpBytes), k_addr, id_g, c > 0);
                mma_commit(&dsempty[b]);
                mma_commit(&kvempty[st]);
                return true;
            };
            for (int c = 0; c < nck && ok; ++c) {
                const int st = c % kStages;
                const uint32_t ph = (c / kStages) & 1;
                ok = mbar_wait(&kvfull[st], ph, abort_flag, p.err) &&
                     mbar_wait(sempty, (c & 1) ^ 1, abort_flag, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(stages + st * 2 * kTile);
                mma_tiles(tmem + kColS, q_addr, k_addr, id_s);           // S  = Q K_c^T
                mma_tiles(tmem + kColDP, o_addr, k_addr + kTile, id_s);  // dP = dO V_c^T
                mma_commit(sfull);
                if (c > 0) ok = issue_dq(c - 1);
            }
            if (ok && issue_dq(nck - 1)) mma_commit(accfull);
        }
    } else {
        // ---------------- workers: thread = query row ----------------
        // two warps per TMEM lane quarter; warp half h owns key columns
        // [64h, 64h + 64) of every chunk
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int q = quarter * 32 + lane;
        const int qq = a0 + q;
        const float xscale = p.scale * kLog2e;
        float l2 = INFINITY, dl = 0.f;
        const long long row = (long long)bh * g.n + r + (long long)g.s * qq;
        if (qq < nr) {
            l2 = *GP(g.bnd, p.lse + row) * kLog2e;
            dl = *GP(g.bnd, p.delta + row);
        }
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        bool ok = true;
        for (int c = 0; c < nck; ++c) {
            const int b = c & 1;
            const uint32_t bph = (c >> 1) & 1;
            const int kbase = kb_lo + c * kB;
            const int jlo = max(qq - g.w - kbase, 0);
            const int jhi = min(min(qq + g.wu, kb_hi) - kbase, kB - 1);
            const bool q_ok = qq < nr;
            const bool full = __all_sync(0xffffffffu, q_ok && jlo <= 64 * half && jhi >= 64 * half + 63);
            bool w_ok = mbar_wait(sfull, c & 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
            tc_fence_after();
            w_ok = mbar_wait(&dsempty[b], bph ^ 1, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
            const uint32_t dsa = smem_u32(ds_op + b * kOpBytes);
#pragma unroll 1
            for (int grp = 2 * half; grp < 2 * half + 2; ++grp) {
                uint32_t sv[32], dv[32];
                tmem_ld32(lane_base + kColS + grp * 32, sv);
                tmem_ld32(lane_base + kColDP + grp * 32, dv);
                tmem_ld_wait();
                uint32_t dk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float ds[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float y = fmaf(__uint_as_float(sv[2 * i + h]), xscale, -l2);
                        if (!full) {
                            const int j = grp * 32 + 2 * i + h;
                            if (!q_ok || j < jlo || j > jhi) y = -INFINITY;
                        }
                        ds[h] = ex2(y) * (__uint_as_float(dv[2 * i + h]) - dl);
                    }
                    dk[i] = pack2<T>(ds[0], ds[1]);
                }
                store_op_row(dsa, q, grp, dk);
            }
            tc_fence_before();
            mbar_arrive(sempty);
            fence_proxy_async_smem();
            mbar_arrive(&dsfull[b]);
        }
        const bool acc_ok = ok && mbar_wait(accfull, 0, abort_flag, p.err);
        if (__all_sync(0xffffffffu, acc_ok)) {
            tc_fence_after();
            T *dst_row = reinterpret_cast<T *>(p.dQ) + row * 64;
            {
                const int h = half;  // channels [32h, 32h + 32)
                uint32_t v[32];
                tmem_ld32(lane_base + kColDQ + h * 32, v);
                tmem_ld_wait();
                if (qq < nr) {
                    const float mul = p.scale;
                    uint4 *o4 = reinterpret_cast<uint4 *>(dst_row + h * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *GP(g.bnd, o4 + u) = make_uint4(
                            pack2<T>(mul * __uint_as_float(v[8 * u]), mul * __uint_as_float(v[8 * u + 1])),
                            pack2<T>(mul * __uint_as_float(v[8 * u + 2]), mul * __uint_as_float(v[8 * u + 3])),
                            pack2<T>(mul * __uint_as_float(v[8 * u + 4]), mul * __uint_as_float(v[8 * u + 5])),
                            pack2<T>(mul * __uint_as_float(v[8 * u + 6]), mul * __uint_as_float(v[8 * u + 7])));
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
// One-pass backward: dK, dV and dQ from one persistent kernel.
// Tile = 128 keys of one residue; for each 128-query chunk of its band:
//   S^T = K Q_c^T, dP^T = V dO_c^T               (tcgen05, TMEM lane = key)
//   P^T, dS^T per key row (8 softmax warps: 2 per TMEM lane quarter, each
//   owning 64 query columns): P^T into tensor memory (packed 16-bit pairs),
//   dS^T as a K-major 128-B-swizzled shared-memory operand
//   dV += P^T dO_c (A from TMEM), dK += dS^T Q_c   (TMEM, lane = key)
//   dQ_c = dS K: the dS^T tile read as an MN-major A operand (M = queries),
//   the K tile as an MN-major B operand, into a TMEM buffer (lane = query).
//   One chunk later the softmax warps copy dQ_c into a swizzled fp32
//   staging tile and a reducer warp adds it into the fp32 accumulator with
//   two TMA reduce-add stores (the final scale and rounding happen in
//   k_bwd_dq_out).  The chunk sequence runs on across tile boundaries: a
//   tile's dV and dK are read out of TMEM during the next tile's first chunk,
//   once its products are done.  K is double-buffered across tiles (dQ of a
//   tile's last chunk still reads it while the next tile's scores are
//   computed); V, read only by the dP^T product, has one buffer that is
//   reloaded after the tile's last dP^T; Q and dO chunks use a 3-stage ring,
//   so each chunk's load has a whole gradient phase to land.
// Each softmax warp loads the lse and delta of its 64 query columns itself
// (two of each per lane, one chunk ahead) and shares them through a per-warp
// shared slot.  Eight softmax warps (two per scheduler, beside the producer,
// MMA and reducer warps) leave each thread 168 registers and the MMA warp's
// scheduler two busy warps to share with.
// The accumulation order of dQ across key tiles is not fixed, so dQ may
// differ in the last bits between runs; dK and dV have one writer per row.
// ---------------------------------------------------------------------------
namespace fused {
constexpr int kParts = 2;                       // 64 query columns per softmax warp
constexpr int kWorkerWarps = 4 * kParts;        // 8
constexpr int kReducerWarp = 2 + kWorkerWarps;  // 10
constexpr int kThreads = 32 * (kReducerWarp + 1);
constexpr int kQS = 2 * kTile;                  // Q and dO of a query chunk: 32 KB
constexpr int kQStages = 3;
constexpr int kStage = 128 * 64 * 4;            // fp32 dQ staging: two 128 x 32 swizzled halves
constexpr int kSlot = 2 * 64 * 4;               // per softmax warp: lse*log2e, delta of 64 queries
constexpr int kSmem = 3 * kTile + kQStages * kQS + kOpBytes + kStage + kWorkerWarps * kSlot + 1024 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384, kColP = 448;

struct KTile {
    int a0, r, bh, nr, qb_lo, qb_hi, nck;
};

__device__ __forceinline__ bool decode_ktile(const Geom &g, int t, int xt, KTile &tl) {
    tl.a0 = (t % xt) * kB;
    const int rest = t / xt;
    tl.r = rest % g.s;
    tl.bh = rest / g.s;
    tl.nr = residue_len(g.n, g.s, tl.r);
    if (tl.a0 >= tl.nr) return false;
    // key b is attended by the queries a with b in [a - w, a + w_upper]
    tl.qb_lo = max(tl.a0 - g.wu, 0);
    tl.qb_hi = min(tl.a0 + kB - 1 + g.w, tl.nr - 1);
    tl.nck = (tl.qb_hi - tl.qb_lo + kB) / kB;
    return true;
}
}  // namespace fused

// kMode 0: the band.  kMode 1: the band with global tokens -- global keys and
// global queries are left out (a local row's global keys and a global row's
// keys are attended through their own columns and rows), and the dK, dV drain
// adds the global rows' terms (a.gdK, a.gdV, every key) and, at a global key,
// the global columns' terms (a.cdK, a.cdV).  kMode 2: the global columns --
// one "key tile" per slice holding the G global keys (gathered, zero past G;
// mapK / mapV over [BH, 128, 64]) against every local query (chunks over the
// whole sequence, stride 1); dQ is added into the accumulator as in the band
// pass and the tile's dK (scaled), dV are written to a.cdK, a.cdV.
template <typename T, bool kBias, bool kDrop, int kMode = 0>
__global__ void __launch_bounds__(fused::kThreads, 1)
    k_bwd_fused(const __grid_constant__ TmapSet mapQ, const __grid_constant__ TmapSet mapK,
                const __grid_constant__ TmapSet mapV, const __grid_constant__ TmapSet mapdO,
                const __grid_constant__ TmapSet mapAcc, const BwdArgs p,
                const __grid_constant__ GlobArgs gl) {
    using namespace fused;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *kbuf = base;                       // [2] K tiles
    uint8_t *vbuf = kbuf + 2 * kTile;           // V tile
    uint8_t *qsbuf = vbuf + kTile;              // [kQStages] query chunks: Q at +0, dO at +kTile
    uint8_t *dst_op = qsbuf + kQStages * kQS;   // dS^T [128 keys x 128 queries]
    uint8_t *stage = dst_op + kOpBytes;         // fp32 dQ: channels [0,32) at +0, [32,64) at +16 KB
    float *slots = reinterpret_cast<float *>(stage + kStage);  // [8 warps][lse | delta][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(slots + kWorkerWarps * (kSlot / 4));
    uint64_t *kfull = bars;            // [2]
    uint64_t *kempty = kfull + 2;      // [2]
    uint64_t *vfull = kempty + 2;      // 1
    uint64_t *vempty = vfull + 1;      // 1
    uint64_t *qfull = vempty + 1;      // [kQStages]
    uint64_t *qempty = qfull + kQStages;  // [kQStages]
    uint64_t *sfull = qempty + kQStages;  // 1
    uint64_t *sempty = sfull + 1;      // 1, count fused::kWorkerWarps
    uint64_t *opfull = sempty + 1;     // 1, count fused::kWorkerWarps
    uint64_t *opempty = opfull + 1;    // 1 (also: dQ of that chunk is in TMEM)
    uint64_t *stfull = opempty + 1;    // 1, count fused::kWorkerWarps
    uint64_t *stempty = stfull + 1;    // 1
    uint64_t *mmadone = stempty + 1;   // 1
    uint64_t *drain = mmadone + 1;     // a flag word that is never set
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *no_abort = reinterpret_cast<volatile int *>(drain);

    // global tokens: bit j of gbits marks position j as global
    uint32_t *gbits = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(bars) + 1024);

    const Geom &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gtiles = (gl.G + kB - 1) / kB;   // kMode 2: key tiles of gathered global keys per slice
    const int xt = kMode == 2 ? 1 : (g.nsub + kB - 1) / kB;
    const int ntiles = kMode == 2 ? g.BH * gtiles : xt * g.s * g.BH;

    if constexpr (kMode != 0) {
        for (int w = threadIdx.x; w < (g.n + 31) / 32; w += fused::kThreads) gbits[w] = 0u;
        __syncthreads();
        for (int k = threadIdx.x; k < gl.G; k += fused::kThreads)
            atomicOr(&gbits[gl.idx[k] >> 5], 1u << (gl.idx[k] & 31));
        // visible to every thread after the barrier below
    }
    auto is_global = [&](int pos) -> bool { return (gbits[pos >> 5] >> (pos & 31)) & 1u; };
    // tile t: kMode 2 has ceil(G / 128) tiles per slice, their keys the
    // gathered global keys and their queries the whole sequence
    auto decode = [&](int t, KTile &tl) -> bool {
        if constexpr (kMode == 2) {
            tl.a0 = (t % gtiles) * kB;
            tl.r = 0;
            tl.bh = t / gtiles;
            tl.nr = g.n;
            tl.qb_lo = 0;
            tl.qb_hi = g.n - 1;
            tl.nck = (g.n + kB - 1) / kB;
            return true;
        } else {
            return decode_ktile(g, t, xt, tl);
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
        }
        mbar_init(vfull, 1);
        mbar_init(vempty, 1);
        mbar_init(sfull, 1);
        mbar_init(sempty, fused::kWorkerWarps);
        mbar_init(opfull, fused::kWorkerWarps);
        mbar_init(opempty, 1);
        mbar_init(stfull, fused::kWorkerWarps);
        mbar_init(stempty, 1);
        mbar_init(mmadone, 1);
        *no_abort = 0;
        *abort_flag = 0;
        fence_barrier_init();
    }
    pdl_trigger();   // the dQ rounding may be scheduled (it waits for this grid)
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------- producer (warp-uniform; lane 0 issues the copies) ----------------
        uint32_t gc = 0, it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            KTile tl;
            if (!decode(t, tl)) continue;
            const CUtensorMap *mq = &mapQ.m[tl.r], *mk = &mapK.m[tl.r], *mv = &mapV.m[tl.r],
                              *mo = &mapdO.m[tl.r];
            const int tb = it & 1;
            // K: buffer tb was last read by the last products of tile it-2;
            // V: its one buffer was last read by the last dP^T of tile it-1
            if (!__all_sync(0xffffffffu, mbar_wait(&kempty[tb], ((it >> 1) & 1) ^ 1, abort_flag, p.err) &&
                                             mbar_wait(vempty, (it & 1) ^ 1, abort_flag, p.err)))
                break;
            if (lane == 0) {
                tma_prefetch_desc(mq);
                tma_prefetch_desc(mk);
                tma_prefetch_desc(mv);
                tma_prefetch_desc(mo);
                mbar_arrive_expect_tx(&kfull[tb], kTile);
                tma_load_dense(kbuf + tb * kTile, mk, &kfull[tb], tl.a0, tl.bh, g.h, g.rs_p != 0);
                mbar_arrive_expect_tx(vfull, kTile);
                tma_load_dense(vbuf, mv, vfull, tl.a0, tl.bh, g.h, g.rs_p != 0);
                // the next tile's K and V into L2: V is reloaded within one
                // gradient phase at the tile boundary
                for (int t2 = t + gridDim.x; t2 < ntiles; t2 += gridDim.x) {
                    KTile nx;
                    if (!decode(t2, nx)) continue;
                    tma_prefetch_dense(&mapK.m[nx.r], nx.a0, nx.bh, g.h, g.rs_p != 0);
                    tma_prefetch_dense(&mapV.m[nx.r], nx.a0, nx.bh, g.h, g.rs_p != 0);
                    break;
                }
            }
            __syncwarp();
            ++it;
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int qs = gc % kQStages;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&qempty[qs], ((gc / kQStages) & 1) ^ 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int qbase = tl.qb_lo + c * kB;
                    mbar_arrive_expect_tx(&qfull[qs], kQS);
                    tma_load_dense(qsbuf + qs * kQS, mq, &qfull[qs], qbase, tl.bh, g.h, g.rs_p != 0);
                    tma_load_dense(qsbuf + qs * kQS + kTile, mo, &qfull[qs], qbase, tl.bh, g.h,
                                   g.rs_o != 0);
                }
                __syncwarp();
            }
        }
        // every copy issued lands before the CTA may exit
        for (uint32_t k = it > 2u ? it - 2 : 0; k < it; ++k)
            mbar_wait(&kfull[k & 1], (k >> 1) & 1, no_abort, nullptr, 100000000ull);
        if (it > 0) mbar_wait(vfull, (it - 1) & 1, no_abort, nullptr, 100000000ull);
        for (uint32_t k = gc > (uint32_t)kQStages ? gc - kQStages : 0; k < gc; ++k)
            mbar_wait(&qfull[k % kQStages], (k / kQStages) & 1, no_abort, nullptr, 100000000ull);
    } else if (warp == 1) {
        // ---------------- MMA issuer (warp-uniform; lane 0 issues) ----------------
        constexpr bool kBf16 = !std::is_same<T, __half>::value;
        constexpr uint32_t id_s = idesc_f16(kB, kB, kBf16, false, false);  // S^T, dP^T
        constexpr uint32_t id_g = idesc_f16(kB, 64, kBf16, false, true);   // dV, dK
        constexpr uint32_t id_q = idesc_f16(kB, 64, kBf16, true, true);    // dQ
        // descriptors of buffer 0; a buffer / K step adds (bytes >> 4)
        const uint64_t d_k = sdesc_sw128(smem_u32(kbuf), 16, 1024);            // K, K-major
        const uint64_t d_v = sdesc_sw128(smem_u32(vbuf), 16, 1024);            // V, K-major
        const uint64_t d_kmn = sdesc_sw128(smem_u32(kbuf), 1024, 1024);        // K as MN-major B
        const uint64_t d_q = sdesc_sw128(smem_u32(qsbuf), 16, 1024);           // Q, K-major
        const uint64_t d_o = sdesc_sw128(smem_u32(qsbuf + kTile), 16, 1024);   // dO, K-major
        const uint64_t d_qmn = sdesc_sw128(smem_u32(qsbuf), 1024, 1024);       // Q as MN-major B
        const uint64_t d_omn = sdesc_sw128(smem_u32(qsbuf + kTile), 1024, 1024);  // dO as MN-major B
        const uint64_t d_dst = sdesc_sw128(smem_u32(dst_op), 16, 1024);        // dS^T, K-major A
        // dS^T read as dS (M = queries): 64-query blocks kOpBytes/2 apart,
        // 8-key groups 1024 B apart
        const uint64_t d_dsmn = sdesc_sw128(smem_u32(dst_op), kOpBytes / 2, 1024);
        auto issue_grad = [&](uint32_t gg, bool first, bool last, int tb, uint32_t itt) -> bool {
            const int qs = gg % kQStages;
            const uint64_t qoff = (uint64_t)((qs * kQS) >> 4), toff = (uint64_t)((tb * kTile) >> 4);
            // the chunk's operand descriptors, formed before the waits so that
            // the 24 products issue back to back
            uint64_t dv_b[8], dk_a[8], dk_b[8], dq_a[8], dq_b[8];
#pragma unroll
            for (int k = 0; k < kB / 16; ++k) {
                // K step k = queries 16k.. (dV, dK) or keys 16k.. (dQ)
                const uint64_t aop = (uint64_t)((((k >> 2) * (kOpBytes / 2)) + (k & 3) * 32) >> 4);
                const uint64_t rows = (uint64_t)((2048 * k) >> 4);
                dv_b[k] = d_omn + qoff + rows;
                dk_a[k] = d_dst + aop;
                dk_b[k] = d_qmn + qoff + rows;
                dq_a[k] = d_dsmn + rows;
                dq_b[k] = d_kmn + toff + rows;
                asm volatile("" ::"l"(dv_b[k]), "l"(dk_b[k]), "l"(dq_b[k]));
            }
            const uint32_t acc0 = first ? 0u : 1u;
            // opfull (phase gg) also says that the softmax warps have read
            // dQ of chunk gg-1 and, in a tile's first chunk, the previous
            // tile's dV and dK out of TMEM: they do so before they arrive
            if (!__all_sync(0xffffffffu, mbar_wait(opfull, gg & 1, abort_flag, p.err))) return false;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kB / 16; ++k) {
                    const uint32_t acc = k == 0 ? acc0 : 1u;
                    mma_f16_ts(tmem + kColDV, tmem + kColP + 8 * k, dv_b[k], id_g, acc);
                    mma_f16_ss(tmem + kColDK, dk_a[k], dk_b[k], id_g, acc);
                    mma_f16_ss(tmem + kColDQ, dq_a[k], dq_b[k], id_q, k > 0 ? 1u : 0u);
                }
                mma_commit(opempty);   // also: dV, dK of the tile are complete after its last chunk
                mma_commit(&qempty[qs]);
                if (last) mma_commit(&kempty[tb]);
            }
            __syncwarp();
            return true;
        };
        uint32_t gc = 0, it = 0, prev = 0, prev_it = 0;
        int prev_tb = 0;
        bool ok = true, have_prev = false, prev_first = false, prev_last = false;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            KTile tl;
            if (!decode(t, tl)) continue;
            const int tb = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&kfull[tb], (it >> 1) & 1, abort_flag, p.err) &&
                                             mbar_wait(vfull, it & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            const uint64_t toff = (uint64_t)((tb * kTile) >> 4);
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int qs = gc % kQStages;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&qfull[qs], (gc / kQStages) & 1, abort_flag, p.err) &&
                                    mbar_wait(sempty, (gc & 1) ^ 1, abort_flag, p.err));
                if (!ok) break;
                tc_fence_after();
                const uint64_t qoff = (uint64_t)((qs * kQS) >> 4);
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ss(tmem + kColS, d_k + toff + 2 * k, d_q + qoff + 2 * k, id_s, k > 0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ss(tmem + kColDP, d_v + 2 * k, d_o + qoff + 2 * k, id_s, k > 0);
                    if (c == tl.nck - 1) mma_commit(vempty);   // the tile's last read of V
                    mma_commit(sfull);
                }
                __syncwarp();
                if (have_prev && !issue_grad(prev, prev_first, prev_last, prev_tb, prev_it)) {
                    ok = false;
                    break;
                }
                have_prev = true;
                prev = gc;
                prev_first = c == 0;
                prev_last = c == tl.nck - 1;
                prev_tb = tb;
                prev_it = it;
            }
            ++it;
        }
        if (ok && have_prev) issue_grad(prev, prev_first, prev_last, prev_tb, prev_it);
        if (lane == 0) mma_commit(mmadone);
        __syncwarp();
        mbar_wait(mmadone, 0, no_abort, nullptr, 100000000ull);
    } else if (warp == kReducerWarp) {
        // ---------------- reducer: staged dQ tiles into the accumulator ----------------
        pdl_wait();   // the row-sum kernel has cleared the accumulator
        uint32_t gc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            KTile tl;
            if (!decode(t, tl)) continue;
            const CUtensorMap *ma = &mapAcc.m[tl.r];
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                if (!__all_sync(0xffffffffu, mbar_wait(stfull, gc & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int qbase = tl.qb_lo + c * kB;
                    tma_reduce_add_3d(ma, stage, 0, qbase, tl.bh);
                    tma_reduce_add_3d(ma, stage + kStage / 2, 32, qbase, tl.bh);
                    bulk_commit();
                    bulk_wait_read();
                    mbar_arrive(stempty);
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else {
        // ---------------- softmax warps: thread = key row ----------------
        pdl_wait();   // the row sums delta are written
        const int quarter = warp & 3;
        const int part = (warp - 2) >> 2;        // query columns [64 part, 64 part + 64)
        const int m = quarter * 32 + lane;       // TMEM lane: key of the tile / query of a dQ chunk
        const float xscale = p.scale * kLog2e;
        const float dscale = 256.f / (256.f - (float)g.drop_t);   // kept values' scale
        const uint32_t lane_base = tmem_addr(tmem, quarter * 32, 0);
        // dS^T: the part's 64 queries are one 64-query block of the operand;
        // fp32 dQ staging: the part's 32 channels are one half of the tile
        const uint32_t drow = smem_u32(dst_op) + part * (kOpBytes / 2) + m * 128;
        const uint32_t srow = smem_u32(stage) + part * (kStage / 2) + m * 128;
        float *slot = slots + (warp - 2) * (kSlot / 4);   // lse (64 queries) | delta (64)
        uint32_t gc = 0, it = 0;
        bool ok = true;
        bool dq_pend = false;   // the dQ of chunk dq_g (in TMEM) waits to be staged
        uint32_t dq_g = 0;
        bool acc_pend = false, acc_ok = false;   // a tile's dV, dK wait to be read out
        unsigned acc_row = 0;   // row bh * n + key of dK, dV (below 2^31); kMode 2: the key's index in G
        int acc_bh = 0;         // kMode 2: the slice
        int acc_gi = -1;        // kMode 1: index in G of a global key, else -1
        // dV (a), dK (b) of key row acc_row, channels [ch0, ch0 + 16)
        auto drain16 = [&](const uint32_t (&a)[16], const uint32_t (&b)[16], int ch0) {
            if constexpr (kMode == 2) {
                // the global columns' dK (scaled), dV of global key acc_row
                // (its index in G) of slice acc_bh, fp32
                if (acc_ok) {
                    float4 *cv = reinterpret_cast<float4 *>(p.cdV + ((size_t)acc_bh * gl.G + acc_row) * 64 + ch0);
                    float4 *ck = reinterpret_cast<float4 *>(p.cdK + ((size_t)acc_bh * gl.G + acc_row) * 64 + ch0);
                    const float sc = p.scale;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = 4 * u;
                        *GP(g.bnd, cv + u) = make_float4(__uint_as_float(a[i]), __uint_as_float(a[i + 1]),
                                            __uint_as_float(a[i + 2]), __uint_as_float(a[i + 3]));
                        *GP(g.bnd, ck + u) = make_float4(sc * __uint_as_float(b[i]), sc * __uint_as_float(b[i + 1]),
                                            sc * __uint_as_float(b[i + 2]), sc * __uint_as_float(b[i + 3]));
                    }
                }
                return;
            }
            if constexpr (kMode == 1) {
                // the global rows' terms (every key) and, at a global key, the
                // global columns' terms, added before the one rounding
                if (acc_ok) {
                    const float sc = p.scale;
                    const size_t goff = (size_t)acc_row * 64 + ch0;   // contiguous layout
                    const uint4 *gv = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.gdV) + goff);
                    const uint4 *gk = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.gdK) + goff);
                    float fv[16], fk[16];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint4 wv = *GP(g.bnd, gv + u), wk = *GP(g.bnd, gk + u);
                        const uint32_t v32[4] = {wv.x, wv.y, wv.z, wv.w}, k32[4] = {wk.x, wk.y, wk.z, wk.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            fv[8 * u + 2 * e] = __uint_as_float(a[8 * u + 2 * e]) + lo16<T>(v32[e]);
                            fv[8 * u + 2 * e + 1] = __uint_as_float(a[8 * u + 2 * e + 1]) + hi16<T>(v32[e]);
                            fk[8 * u + 2 * e] = fmaf(sc, __uint_as_float(b[8 * u + 2 * e]), lo16<T>(k32[e]));
                            fk[8 * u + 2 * e + 1] = fmaf(sc, __uint_as_float(b[8 * u + 2 * e + 1]), hi16<T>(k32[e]));
                        }
                    }
                    if (acc_gi >= 0) {
                        const float *cv = p.cdV + ((size_t)acc_bh * gl.G + acc_gi) * 64 + ch0;
                        const float *ck = p.cdK + ((size_t)acc_bh * gl.G + acc_gi) * 64 + ch0;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            fv[i] += *GP(g.bnd, cv + i);
                            fk[i] += *GP(g.bnd, ck + i);
                        }
                    }
                    uint4 *v4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.dV) + goff);
                    uint4 *k4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.dK) + goff);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int i = 8 * u;
                        *GP(g.bnd, v4 + u) = make_uint4(pack2<T>(fv[i], fv[i + 1]), pack2<T>(fv[i + 2], fv[i + 3]),
                                           pack2<T>(fv[i + 4], fv[i + 5]), pack2<T>(fv[i + 6], fv[i + 7]));
                        *GP(g.bnd, k4 + u) = make_uint4(pack2<T>(fk[i], fk[i + 1]), pack2<T>(fk[i + 2], fk[i + 3]),
                                           pack2<T>(fk[i + 4], fk[i + 5]), pack2<T>(fk[i + 6], fk[i + 7]));
                    }
                }
                return;
            }
            if (acc_ok) {
                const long long off = dense_row(g, acc_row, g.rs_p) + ch0;
                uint4 *v4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.dV) + off);
                uint4 *k4 = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.dK) + off);
                const float sc = p.scale;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int i = 8 * u;
                    *GP(g.bnd, v4 + u) = make_uint4(pack2<T>(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                                       pack2<T>(__uint_as_float(a[i + 2]), __uint_as_float(a[i + 3])),
                                       pack2<T>(__uint_as_float(a[i + 4]), __uint_as_float(a[i + 5])),
                                       pack2<T>(__uint_as_float(a[i + 6]), __uint_as_float(a[i + 7])));
                    *GP(g.bnd, k4 + u) = make_uint4(pack2<T>(sc * __uint_as_float(b[i]), sc * __uint_as_float(b[i + 1])),
                                       pack2<T>(sc * __uint_as_float(b[i + 2]), sc * __uint_as_float(b[i + 3])),
                                       pack2<T>(sc * __uint_as_float(b[i + 4]), sc * __uint_as_float(b[i + 5])),
                                       pack2<T>(sc * __uint_as_float(b[i + 6]), sc * __uint_as_float(b[i + 7])));
                }
            }
        };
        // dV, dK of key row acc_row (channels [32 part, +32)) out of TMEM
        // into dV, dK; the caller has waited for the tile's last products
        auto drain_acc = [&]() {
            uint32_t a0[16], b0[16], a1[16], b1[16];
            tmem_ld16(lane_base + kColDV + 32 * part, a0);
            tmem_ld16(lane_base + kColDK + 32 * part, b0);
            tmem_ld16(lane_base + kColDV + 32 * part + 16, a1);
            tmem_ld16(lane_base + kColDK + 32 * part + 16, b1);
            tmem_ld_wait();
            drain16(a0, b0, 32 * part);
            drain16(a1, b1, 32 * part + 16);
        };
        // lse, delta of the queries cb + lane and cb + 32 + lane
        // (with the keep-bit cache, also the cached keep bits of those
        // queries for the warp's 32 keys)
        auto load_rowstats = [&](const KTile &tl, int cb, float (&l)[2], float (&d)[2], uint32_t (&km)[2]) {
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                l[w] = 0.f;
                d[w] = 0.f;
                km[w] = 0u;
                const int qs = cb + 32 * w + lane;
                if (qs < tl.nr) {
                    const long long row = (long long)tl.bh * g.n + tl.r + (long long)g.s * qs;
                    l[w] = *GP(g.bnd, p.lse + row);
                    d[w] = *GP(g.bnd, p.delta + row);
                    if (kDrop && g.dmask) {
                        const long long wi =
                            dmask_word(g, tl.bh, tl.r + (long long)g.s * qs, qs, (tl.a0 + 32 * quarter) / 32);
                        if (wi >= 0) km[w] = __ldg(GP(g.bnd, g.dmask + wi));
                    }
                }
            }
        };
        float lq_next[2] = {0.f, 0.f}, dq_next[2] = {0.f, 0.f};
        uint32_t km_next[2] = {0u, 0u};
        // dQ of chunk dq_g (channels [32 part, +32) of query row m) into the
        // staging tile, once the reducer has read the previous one
        auto stage_dq = [&](const uint32_t (&dqv)[32]) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(stempty, (dq_g & 1) ^ 1, abort_flag, p.err))) return false;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                sts16(srow + ((u ^ (m & 7)) << 4),
                      make_uint4(dqv[4 * u], dqv[4 * u + 1], dqv[4 * u + 2], dqv[4 * u + 3]));
            fence_proxy_async_smem();
            mbar_arrive_warp(stfull);
            return true;
        };

        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            KTile tl;
            if (!decode(t, tl)) continue;
            const int kk = tl.a0 + m;
            // key bias of this thread's key (log2 units), the same for every query
            uint64_t kb2 = f2(0.f, 0.f);
            if constexpr (kBias) {
                // the key's position: kMode 2 gathers the global keys (index
                // kk in G; the rows past G are padding)
                const int pos = kMode == 2 ? (kk < gl.G ? gl.idx[kk] : -1) : (kk < tl.nr ? tl.r + g.s * kk : -1);
                if (pos >= 0) {
                    const float kb = __ldg(GP(g.bnd, g.kbias + (size_t)(tl.bh / g.h) * g.n + pos)) * kLog2e;
                    kb2 = f2(kb, kb);
                }
            }
            // kMode 1: a global key takes no band query; kMode 2: the rows past
            // the G gathered keys are padding
            bool key_off = kk >= tl.nr;
            if constexpr (kMode == 1) key_off = key_off || is_global(tl.r + g.s * kk);
            if constexpr (kMode == 2) key_off = kk >= gl.G;
            for (int c = 0; c < tl.nck; ++c, ++gc) {
                const int qbase = tl.qb_lo + c * kB;
                const int cbase = qbase + 64 * part;
                // vm[w]: this key's queries among the columns [32 w, 32 w + 32)
                // of the part (kMode 2: every query of the sequence)
                uint32_t vm[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int cb = cbase + 32 * w;
                    const int jlo = kMode == 2 ? 0 : max(kk - g.wu - cb, 0);
                    const int jhi = kMode == 2 ? min(tl.nr - 1 - cb, 31) : min(min(kk + g.w, tl.nr - 1) - cb, 31);
                    vm[w] = (key_off || jlo > jhi) ? 0u : ((2u << jhi) - 1u) & (0xffffffffu << jlo);
                    if constexpr (kMode != 0) {
                        // global queries (query column `lane` of the word) take no
                        // band or global-column keys: their rows are dense, done apart
                        const int qsub = cb + lane;
                        const bool qg = qsub < tl.nr && is_global(tl.r + g.s * qsub);
                        vm[w] &= ~__ballot_sync(0xffffffffu, qg);
                    }
                }
                const bool full = __all_sync(0xffffffffu, (vm[0] & vm[1]) == 0xffffffffu);
                const bool empty = __all_sync(0xffffffffu, (vm[0] | vm[1]) == 0u);
                // dropout: bit j of keepcol[w] = keep(query column 32 w + j of the
                // part, this key).  Lane l draws the block of query column 32 w + l
                // for the warp's 32 keys (one block: the warp's keys start on a
                // multiple of 32) and a transpose of the warp's 32 x 32 bit
                // matrix hands each key row its bits.
                uint32_t keepcol[2] = {0xffffffffu, 0xffffffffu};
                if constexpr (kDrop) {
                    if (!empty && !g.dmask) {
#pragma unroll
                        for (int w = 0; w < 2; ++w) {
                            unsigned long long wv[4];
                            philox4x64_10((unsigned long long)((tl.a0 + 32 * quarter) / 32),
                                          (unsigned long long)(tl.r + (long long)g.s * (cbase + 32 * w + lane)),
                                          (unsigned long long)tl.bh, 0, g.seed, 0, wv);
                            keepcol[w] = bit_transpose32(keep_bits32(wv, g.drop_t), lane);
                        }
                    }
                }
                // lse and delta of the part's queries: loaded one chunk ahead
                // (the first chunk of a tile here), so that their latency is
                // hidden behind the previous chunk
                float lq[2], dq[2];
                uint32_t km[2];
                if (c == 0) {
                    load_rowstats(tl, cbase, lq, dq, km);
                } else {
                    lq[0] = lq_next[0];
                    lq[1] = lq_next[1];
                    dq[0] = dq_next[0];
                    dq[1] = dq_next[1];
                    km[0] = km_next[0];
                    km[1] = km_next[1];
                }
                if (c + 1 < tl.nck) load_rowstats(tl, cbase + kB, lq_next, dq_next, km_next);
                if constexpr (kDrop) {
                    // the cached keep bits (query column 32 w + lane's word for
                    // the warp's keys), transposed to the key rows
                    if (!empty && g.dmask) {
#pragma unroll
                        for (int w = 0; w < 2; ++w) keepcol[w] = bit_transpose32(km[w], lane);
                    }
                }
                if (!__all_sync(0xffffffffu, mbar_wait(sfull, gc & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                __syncwarp();   // the previous chunk's reads of the slot are done
                slot[lane] = lq[0] * kLog2e;
                slot[32 + lane] = lq[1] * kLog2e;
                slot[64 + lane] = dq[0];
                slot[96 + lane] = dq[1];
                __syncwarp();
                const float4 *l4 = reinterpret_cast<const float4 *>(slot);
                const float4 *d4 = reinterpret_cast<const float4 *>(slot + 64);
                const uint64_t xs2 = f2(xscale, xscale);
                // packed P^T and dS^T of the part's columns: [32 w + 2 q, +2) in
                // word q of pk[w], dk[w]
                uint32_t pk[2][16], dk[2][16];
                // columns [8h, 8h + 8) of the part in eight steps
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const int w = h >> 2;                 // word of the step's columns
                    const uint32_t vmask = vm[w], keep = keepcol[w];
                    uint32_t sv[8], dv[8];
                    tmem_ld8(lane_base + kColS + 64 * part + 8 * h, sv);
                    tmem_ld8(lane_base + kColDP + 64 * part + 8 * h, dv);
                    tmem_ld_wait();
                    if (h == 7) {
                        tc_fence_before();
                        mbar_arrive_warp(sempty);
                    }
                    if (empty) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) pk[w][4 * (h & 3) + i] = dk[w][4 * (h & 3) + i] = 0u;
                        continue;
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float4 lv = l4[2 * h + u], dl = d4[2 * h + u];
                        const int i = 4 * u;                  // within the step
                        const int j = 8 * (h & 3) + i;        // within the word
                        const int q = 4 * (h & 3) + 2 * u;    // packed word of pk[w], dk[w]
                        float p0, p1, p2, p3;
                        {
                            float y0, y1, y2, y3;
                            // x * scale * log2e (+ key bias) - lse * log2e
                            const uint64_t c01 = kBias ? sub2(kb2, f2(lv.x, lv.y)) : f2(-lv.x, -lv.y);
                            const uint64_t c23 = kBias ? sub2(kb2, f2(lv.z, lv.w)) : f2(-lv.z, -lv.w);
                            f2split(fma2(f2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), xs2, c01), y0, y1);
                            f2split(fma2(f2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])), xs2, c23), y2, y3);
                            p0 = ex2(y0);
                            p1 = ex2(y1);
                            p2 = ex2(y2);
                            p3 = ex2(y3);
                        }
                        if (!full) {
                            if (!((vmask >> j) & 1u)) p0 = 0.f;
                            if (!((vmask >> (j + 1)) & 1u)) p1 = 0.f;
                            if (!((vmask >> (j + 2)) & 1u)) p2 = 0.f;
                            if (!((vmask >> (j + 3)) & 1u)) p3 = 0.f;
                        }
                        float s0, s1, s2, s3;
                        if constexpr (kDrop) {
                            // dS = p (f dP - delta), and dV takes p f
                            const float f0 = ((keep >> j) & 1u) ? dscale : 0.f;
                            const float f1 = ((keep >> (j + 1)) & 1u) ? dscale : 0.f;
                            const float f2_ = ((keep >> (j + 2)) & 1u) ? dscale : 0.f;
                            const float f3 = ((keep >> (j + 3)) & 1u) ? dscale : 0.f;
                            f2split(mul2(f2(p0, p1), fma2(f2(f0, f1), f2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])), f2(-dl.x, -dl.y))), s0, s1);
                            f2split(mul2(f2(p2, p3), fma2(f2(f2_, f3), f2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3])), f2(-dl.z, -dl.w))), s2, s3);
                            p0 *= f0;
                            p1 *= f1;
                            p2 *= f2_;
                            p3 *= f3;
                        } else {
                            f2split(mul2(f2(p0, p1), sub2(f2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])), f2(dl.x, dl.y))), s0, s1);
                            f2split(mul2(f2(p2, p3), sub2(f2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3])), f2(dl.z, dl.w))), s2, s3);
                        }
                        pk[w][q] = pack2<T>(p0, p1);
                        pk[w][q + 1] = pack2<T>(p2, p3);
                        dk[w][q] = pack2<T>(s0, s1);
                        dk[w][q + 1] = pack2<T>(s2, s3);
                    }
                }
                // the products of chunk gc-1 are done: its operands are free,
                // its dQ is in TMEM and, at a tile boundary, the previous
                // tile's dV and dK are complete
                if (!__all_sync(0xffffffffu, mbar_wait(opempty, (gc & 1) ^ 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // P^T: query columns [64 part, +64) are TMEM columns [32 part, +32) of the P region
                tmem_st16(lane_base + kColP + 32 * part, pk[0]);
                tmem_st16(lane_base + kColP + 32 * part + 16, pk[1]);
                // dS^T: columns 8u.. of the part are 16-byte chunk u of the key row
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t off = (uint32_t)((u ^ (m & 7)) << 4);
                    const int w = u >> 2, q = 4 * (u & 3);
                    sts16(drow + off, make_uint4(dk[w][q], dk[w][q + 1], dk[w][q + 2], dk[w][q + 3]));
                }
                tmem_st_wait();
                // the previous tile's dV, dK (in its first chunk) and dQ of
                // chunk gc-1 out of TMEM before the operands are signalled:
                // the next products overwrite them
                if (acc_pend) {
                    drain_acc();
                    acc_pend = false;
                }
                uint32_t dqv[32];
                if (dq_pend) {
                    tmem_ld32(lane_base + kColDQ + 32 * part, dqv);
                    tmem_ld_wait();
                }
                tc_fence_before();
                fence_proxy_async_smem();
                mbar_arrive_warp(opfull);
                if (dq_pend && !stage_dq(dqv)) {
                    ok = false;
                    break;
                }
                dq_pend = true;
                dq_g = gc;
            }
            if (!ok) break;
            // dV, dK of these keys: read out during the next chunk (or at the end)
            acc_pend = true;
            acc_ok = kk < tl.nr;
            acc_row = (unsigned)(tl.bh * g.n + tl.r + g.s * kk);
            if constexpr (kMode == 2) {
                acc_ok = kk < gl.G;
                acc_row = (unsigned)kk;
                acc_bh = tl.bh;
            }
            if constexpr (kMode == 1) {
                acc_gi = -1;
                const int pos = tl.r + g.s * kk;
                if (acc_ok && is_global(pos)) {
                    int lo = 0, hi = gl.G - 1;   // the index is sorted
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (gl.idx[mid] < pos) lo = mid + 1;
                        else hi = mid;
                    }
                    acc_gi = lo;
                    acc_bh = tl.bh;
                }
            }
            ++it;
        }
        if (ok && dq_pend) {
            // the last chunk's products (opempty phase gc-1): its dQ and the
            // last tile's dV, dK
            if (__all_sync(0xffffffffu, mbar_wait(opempty, (gc - 1) & 1, abort_flag, p.err))) {
                tc_fence_after();
                if (acc_pend) drain_acc();
                uint32_t dqv[32];
                tmem_ld32(lane_base + kColDQ + 32 * part, dqv);
                tmem_ld_wait();
                tc_fence_before();
                stage_dq(dqv);
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
// exact fp32 path: one CTA per row, one thread per channel; the backward of the
// fp32 fused forward, recomputing each slot's probability from lse.
//   dQ pass (rows = queries), then dK / dV pass (rows = keys).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_dot(float x, float *part) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (lane == 0) part[wid] = x;
    __syncthreads();
    float s = 0.f;
    for (int k = 0; k < nw; ++k) s += part[k];
    __syncthreads();
    return s;
}

__global__ void __launch_bounds__(128) k_bwd_f32(const BwdArgs p, int pass) {
    const Geom &g = p.g;
    const long long R = blockIdx.x;
    const int x = (int)(R % g.n);
    const long long bh = R / g.n;
    const int c = threadIdx.x;
    __shared__ float part[4];
    // row y of the slice is at y * ps (Q, K, V) or y * os (dO) from row 0
    const long long ps = g.rs_p ? g.rs_p : g.hd, os = g.rs_o ? g.rs_o : g.hd;
    const float *Q = reinterpret_cast<const float *>(p.Q) + dense_row(g, bh * g.n, g.rs_p);
    const float *K = reinterpret_cast<const float *>(p.K) + dense_row(g, bh * g.n, g.rs_p);
    const float *V = reinterpret_cast<const float *>(p.V) + dense_row(g, bh * g.n, g.rs_p);
    const float *dO = reinterpret_cast<const float *>(p.dO) + dense_row(g, bh * g.n, g.rs_o);
    const float *lse = p.lse + bh * g.n;
    const float *delta = p.delta + bh * g.n;
    const bool on = c < g.hd;
    float acc_a = 0.f, acc_b = 0.f;
    for (int t = 0; t < g.D; ++t) {
        // pass 0: x is the query, the key is j;  pass 1: x is the key, the query is i
        const long long y = pass == 0 ? (long long)x + (long long)(t - g.w) * g.s
                                      : (long long)x - (long long)(t - g.w) * g.s;
        if (y < 0 || y >= g.n) continue;
        const long long i = pass == 0 ? x : y, j = pass == 0 ? y : x;
        const float sdot = block_dot(on ? *GP(g.bnd, Q + i * ps + c) * *GP(g.bnd, K + j * ps + c) : 0.f, part);
        const float pdot = block_dot(on ? *GP(g.bnd, dO + i * os + c) * *GP(g.bnd, V + j * ps + c) : 0.f, part);
        const float kb = g.kbias ? *GP(g.bnd, g.kbias + (size_t)(bh / g.h) * g.n + (size_t)j) : 0.f;
        const float pr = expf(p.scale * sdot + kb - *GP(g.bnd, lse + i));
        const float f = drop_factor(g, bh, i, j);   // dropout keep-and-scale factor
        const float ds = pr * (f * pdot - *GP(g.bnd, delta + i));
        if (!on) continue;
        if (pass == 0) {
            acc_a = fmaf(ds, *GP(g.bnd, K + j * ps + c), acc_a);
        } else {
            acc_a = fmaf(ds, *GP(g.bnd, Q + i * ps + c), acc_a);   // dK
            acc_b = fmaf(pr * f, *GP(g.bnd, dO + i * os + c), acc_b);  // dV
        }
    }
    if (!on) return;
    const long long out = dense_row(g, R, g.rs_p) + c;
    if (pass == 0) {
        *GP(g.bnd, reinterpret_cast<float *>(p.dQ) + out) = p.scale * acc_a;
    } else {
        *GP(g.bnd, reinterpret_cast<float *>(p.dK) + out) = p.scale * acc_a;
        *GP(g.bnd, reinterpret_cast<float *>(p.dV) + out) = acc_b;
    }
}

__global__ void __launch_bounds__(128) k_bwd_delta_f32(const BwdArgs p) {
    const long long R = blockIdx.x;
    const int c = threadIdx.x;
    __shared__ float part[4];
    const float *O = reinterpret_cast<const float *>(p.O) + dense_row(p.g, R, p.g.rs_o);
    const float *dO = reinterpret_cast<const float *>(p.dO) + dense_row(p.g, R, p.g.rs_o);
    const float v = block_dot(c < p.g.hd ? *GP(p.g.bnd, O + c) * *GP(p.g.bnd, dO + c) : 0.f, part);
    if (c == 0) *GP(p.g.bnd, p.delta + R) = v;
}

template <typename T>
cudaError_t launch_t(const TmapSet &mq, const TmapSet &mk, const TmapSet &mv, const TmapSet &mo,
                     const BwdArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    const long long per_block = 8LL * kDeltaRowsPerWarp;
    k_bwd_delta<T><<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int tiles = (a.g.nsub + kB - 1) / kB;
    dim3 grid(tiles, a.g.s, a.g.BH);
    e = ensure_smem(reinterpret_cast<const void *>(k_bwd_dkdv<T>), kSmemDKDV);
    if (e != cudaSuccess) return e;
    k_bwd_dkdv<T><<<grid, kThreads, kSmemDKDV, st>>>(mq, mk, mv, mo, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = ensure_smem(reinterpret_cast<const void *>(k_bwd_dq<T>), kSmemDQ);
    if (e != cudaSuccess) return e;
    k_bwd_dq<T><<<grid, kThreads, kSmemDQ, st>>>(mq, mk, mv, mo, a);
    return cudaGetLastError();
}

template <typename T, bool kBias, bool kDrop>
cudaError_t launch_fused_t(const TmapSet &mq, const TmapSet &mk, const TmapSet &mv, const TmapSet &mo,
                           const TmapSet &macc, const BwdArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    const long long per_block = 8LL * kDeltaRowsPerWarp;
    k_bwd_delta<T><<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)((a.g.nsub + kB - 1) / kB) * a.g.s * a.g.BH;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = (int)(tiles < sms ? tiles : sms);
    e = ensure_smem(reinterpret_cast<const void *>(k_bwd_fused<T, kBias, kDrop>), fused::kSmem);
    if (e != cudaSuccess) return e;
    // the one-pass kernel and the dQ rounding start early (programmatic
    // dependent launch) and wait inside for what the kernel before wrote
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(fused::kThreads);
    cfg.dynamicSmemBytes = fused::kSmem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    GlobArgs none;
    none.G = 0;
    e = cudaLaunchKernelEx(&cfg, k_bwd_fused<T, kBias, kDrop>, mq, mk, mv, mo, macc, a, none);
    if (e != cudaSuccess) return e;
    const long long groups = rows * 8;
    cfg.gridDim = dim3((unsigned)((groups + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, k_bwd_dq_out<T>, a);
}

// ---------------------------------------------------------------------------
// global tokens: gather the G global rows of Q, O, dO, lse into compact
// buffers (the global rows' backward) and the global keys / values into
// ceil(G / 128) [128, 64] tiles per slice, zero past G (the global columns'
// "key tiles").
// Contiguous layout; one CTA per slice.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) k_glob_gather(const BwdArgs p, const __grid_constant__ GlobArgs gl,
                                                     const GlobBwdBufs gb) {
    const long long bh = blockIdx.x;
    const int n = p.g.n, G = gl.G;
    const uint4 *K4 = reinterpret_cast<const uint4 *>(p.K), *V4 = reinterpret_cast<const uint4 *>(p.V);
    const uint4 *Q4 = reinterpret_cast<const uint4 *>(p.Q), *O4 = reinterpret_cast<const uint4 *>(p.O);
    const uint4 *dO4 = reinterpret_cast<const uint4 *>(p.dO);
    uint4 *KG4 = reinterpret_cast<uint4 *>(gb.KG), *VG4 = reinterpret_cast<uint4 *>(gb.VG);
    const int grows = (G + kB - 1) / kB * kB;   // whole 128-key tiles
    for (int i = threadIdx.x; i < grows * 8; i += blockDim.x) {
        const int row = i >> 3, c = i & 7;   // 8 x 16 bytes per 64-element row
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (row < G) {
            const size_t src = ((size_t)bh * n + gl.idx[row]) * 8 + c;
            kv = *GP(p.g.bnd, K4 + src);
            vv = *GP(p.g.bnd, V4 + src);
        }
        *GP(p.g.bnd, KG4 + ((size_t)bh * grows + row) * 8 + c) = kv;
        *GP(p.g.bnd, VG4 + ((size_t)bh * grows + row) * 8 + c) = vv;
    }
    uint4 *Qg4 = reinterpret_cast<uint4 *>(gb.Qg), *Og4 = reinterpret_cast<uint4 *>(gb.Og);
    uint4 *dOg4 = reinterpret_cast<uint4 *>(gb.dOg);
    for (int i = threadIdx.x; i < G * 8; i += blockDim.x) {
        const int row = i >> 3, c = i & 7;
        const size_t src = ((size_t)bh * n + gl.idx[row]) * 8 + c, dst = ((size_t)bh * G + row) * 8 + c;
        *GP(p.g.bnd, Qg4 + dst) = *GP(p.g.bnd, Q4 + src);
        *GP(p.g.bnd, Og4 + dst) = *GP(p.g.bnd, O4 + src);
        *GP(p.g.bnd, dOg4 + dst) = *GP(p.g.bnd, dO4 + src);
    }
    for (int k = threadIdx.x; k < G; k += blockDim.x)
        *GP(p.g.bnd, gb.lseg + bh * G + k) = *GP(p.g.bnd, p.lse + bh * n + gl.idx[k]);
}

// the global rows' dQ (computed by the global-query backward) into dQ
__global__ void __launch_bounds__(256) k_glob_dq_rows(const BwdArgs p, const __grid_constant__ GlobArgs gl,
                                                      const void *dQg) {
    const long long bh = blockIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(dQg);
    uint4 *dst = reinterpret_cast<uint4 *>(p.dQ);
    for (int i = threadIdx.x; i < gl.G * 8; i += blockDim.x) {
        const int row = i >> 3, c = i & 7;
        *GP(p.g.bnd, dst + ((size_t)bh * p.g.n + gl.idx[row]) * 8 + c) = *GP(p.g.bnd, src + ((size_t)bh * gl.G + row) * 8 + c);
    }
}

template <typename T, bool kBias>
cudaError_t launch_glob_t(const TmapSet &mq, const TmapSet &mk, const TmapSet &mv, const TmapSet &mo,
                          const TmapSet &macc, const TmapSet &mq1, const TmapSet &mo1, const TmapSet &mkc,
                          const TmapSet &mvc, const TmapSet &macc1, const GlobArgs &gl, const GlobBwdBufs &gb,
                          const BwdArgs &a, const GlobalProjArgs &gp, const TmapSet &gmk, const TmapSet &gmv,
                          const TmapSet &gmq, const TmapSet &gmo, cudaStream_t st) {
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const long long rows = (long long)a.g.BH * a.g.n;
    // 1. delta for every row; the dQ accumulator cleared
    const long long per_block = 8LL * kDeltaRowsPerWarp;
    k_bwd_delta<T><<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. the global rows and the global keys / values gathered
    k_glob_gather<T><<<(unsigned)a.g.BH, 256, 0, st>>>(a, gl, gb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. the global rows: dense attention of the G global queries over every
    //    key (dQ of those rows into gb.dQg, their dK, dV terms into a.gdK, a.gdV)
    if ((e = launch_global_proj_bwd_tc(std::is_same<T, __half>::value ? kF16 : kBF16, gmk, gmv, gmq, gmo, gp, st)) !=
        cudaSuccess)
        return e;
    const size_t smem = fused::kSmem + (size_t)((a.g.n + 31) / 32) * 4;
    // 4. the global columns: every local query against the G global keys
    {
        BwdArgs ac = a;
        ac.g.s = 1;
        ac.g.nsub = a.g.n;
        e = ensure_smem(reinterpret_cast<const void *>(k_bwd_fused<T, kBias, false, 2>), (int)smem);
        if (e != cudaSuccess) return e;
        const int ctiles = a.g.BH * ((gl.G + kB - 1) / kB);
        const int grid = ctiles < sms ? ctiles : sms;
        k_bwd_fused<T, kBias, false, 2><<<grid, fused::kThreads, smem, st>>>(mq1, mkc, mvc, mo1, macc1, ac, gl);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 5. the band (global keys and queries left out), its dK, dV drain adding
    //    the global terms; 6. the dQ rounding -- both programmatic dependents
    const long long tiles = (long long)((a.g.nsub + kB - 1) / kB) * a.g.s * a.g.BH;
    const int grid = (int)(tiles < sms ? tiles : sms);
    e = ensure_smem(reinterpret_cast<const void *>(k_bwd_fused<T, kBias, false, 1>), (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(fused::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_bwd_fused<T, kBias, false, 1>, mq, mk, mv, mo, macc, a, gl);
    if (e != cudaSuccess) return e;
    const long long groups = rows * 8;
    cfg.gridDim = dim3((unsigned)((groups + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    if ((e = cudaLaunchKernelEx(&cfg, k_bwd_dq_out<T>, a)) != cudaSuccess) return e;
    // 7. the global rows' dQ
    k_glob_dq_rows<<<(unsigned)a.g.BH, 256, 0, st>>>(a, gl, gb.dQg);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band_attention_bwd_glob(DType dt, const TmapSet &mq, const TmapSet &mk, const TmapSet &mv,
                                           const TmapSet &mo, const TmapSet &macc, const TmapSet &mq1,
                                           const TmapSet &mo1, const TmapSet &mkc, const TmapSet &mvc,
                                           const TmapSet &macc1, const GlobArgs &gl, const GlobBwdBufs &gb,
                                           const BwdArgs &a, const GlobalProjArgs &gp, const TmapSet &gmk,
                                           const TmapSet &gmv, const TmapSet &gmq, const TmapSet &gmo,
                                           cudaStream_t st) {
    if (!a.dqacc || gl.G < 1 || a.g.BH > 65535) return cudaErrorInvalidValue;
    // with the key bias: its band pass and its global-columns pass
#define SWAB_GLOB_BWD(T, B)                                                                                  \
    launch_glob_t<T, B>(mq, mk, mv, mo, macc, mq1, mo1, mkc, mvc, macc1, gl, gb, a, gp, gmk, gmv, gmq, gmo, st)
    if (dt == kF16) return a.g.kbias ? SWAB_GLOB_BWD(__half, true) : SWAB_GLOB_BWD(__half, false);
    if (dt == kBF16) return a.g.kbias ? SWAB_GLOB_BWD(__nv_bfloat16, true) : SWAB_GLOB_BWD(__nv_bfloat16, false);
#undef SWAB_GLOB_BWD
    return cudaErrorInvalidValue;
}

cudaError_t launch_band_attention_bwd_fused(DType dt, const TmapSet &mq, const TmapSet &mk,
                                            const TmapSet &mv, const TmapSet &mo, const TmapSet &macc,
                                            const BwdArgs &a, cudaStream_t st) {
    if (!a.dqacc) return cudaErrorInvalidValue;
    const int v = (a.g.kbias ? 1 : 0) + (a.g.drop_t > 0 ? 2 : 0);
    if (dt == kF16) {
        switch (v) {
            case 0: return launch_fused_t<__half, false, false>(mq, mk, mv, mo, macc, a, st);
            case 1: return launch_fused_t<__half, true, false>(mq, mk, mv, mo, macc, a, st);
            case 2: return launch_fused_t<__half, false, true>(mq, mk, mv, mo, macc, a, st);
            default: return launch_fused_t<__half, true, true>(mq, mk, mv, mo, macc, a, st);
        }
    }
    switch (v) {
        case 0: return launch_fused_t<__nv_bfloat16, false, false>(mq, mk, mv, mo, macc, a, st);
        case 1: return launch_fused_t<__nv_bfloat16, true, false>(mq, mk, mv, mo, macc, a, st);
        case 2: return launch_fused_t<__nv_bfloat16, false, true>(mq, mk, mv, mo, macc, a, st);
        default: return launch_fused_t<__nv_bfloat16, true, true>(mq, mk, mv, mo, macc, a, st);
    }
}

cudaError_t launch_band_attention_bwd_tc(DType dt, const TmapSet &mq, const TmapSet &mk,
                                         const TmapSet &mv, const TmapSet &mo, const BwdArgs &a,
                                         cudaStream_t st) {
    if (dt == kF16) return launch_t<__half>(mq, mk, mv, mo, a, st);
    return launch_t<__nv_bfloat16>(mq, mk, mv, mo, a, st);
}

cudaError_t launch_band_attention_bwd_f32(const BwdArgs &a, cudaStream_t st) {
    const long long rows = (long long)a.g.BH * a.g.n;
    const int threads = ((a.g.hd + 31) / 32) * 32;
    k_bwd_delta_f32<<<(unsigned)rows, threads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_bwd_f32<<<(unsigned)rows, threads, 0, st>>>(a, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_bwd_f32<<<(unsigned)rows, threads, 0, st>>>(a, 1);
    return cudaGetLastError();
}

}  // namespace swab
