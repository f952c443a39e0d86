// swab_common.cuh -- device helpers shared by the library's kernels:
// problem geometry, element conversions, and inline-PTX wrappers for
// mbarriers, TMA (cp.async.bulk.tensor), and the 5th-generation tensor cores
// (tcgen05 MMA with accumulators in tensor memory).  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/swab.h"

namespace swab {

constexpr int kMaxStride = SWAB_MAX_DILATION + 1;
constexpr int kMaxGlobal = SWAB_MAX_GLOBAL;

// Bits of the device status word (bit k <-> swab_status k).
constexpr unsigned kErrTimeout = 1u << SWAB_ERR_TIMEOUT;
constexpr unsigned kErrBounds = 1u << SWAB_ERR_BOUNDS;

// ---------------------------------------------------------------------------
// Bounds checks (SWAB_BOUNDS_CHECK=1 builds).  Every plain global access of a
// kernel names its address through GP(bounds, pointer) (or GPN with an
// explicit byte count for vector and bulk accesses).  In the regular build
// the macro is the pointer itself.  In the checked build it tests the bytes
// [p, p + size) against the call's buffer extents, which the host writes into
// the kernel arguments; outside all of them the access is redirected to a
// scratch line of the library (a store lands there, a load reads it), the
// status word gets SWAB_ERR_BOUNDS and the first such site is recorded.
// ---------------------------------------------------------------------------
#ifndef SWAB_BOUNDS_CHECK
#define SWAB_BOUNDS_CHECK 0
#endif

constexpr int kBoundsMax = 24;

struct Bounds {
    int n;                                  // extents in use
    unsigned long long lo[kBoundsMax];      // byte ranges [lo, hi)
    unsigned long long hi[kBoundsMax];
    unsigned *err;                          // device status word
    unsigned long long *rec;                // first miss: site + 1, address, bytes
    void *sink;                             // 256-byte scratch line
};

#if SWAB_BOUNDS_CHECK
static __device__ __noinline__ void *bounds_check(const Bounds *b, const void *p, unsigned bytes, unsigned site) {
    const unsigned long long a = reinterpret_cast<unsigned long long>(p);
    for (int k = 0; k < b->n; ++k)
        if (a >= b->lo[k] && a + bytes <= b->hi[k]) return const_cast<void *>(p);
    atomicOr(b->err, kErrBounds);
    if (atomicCAS(b->rec, 0ull, (unsigned long long)site + 1ull) == 0ull) {
        b->rec[1] = a;
        b->rec[2] = bytes;
    }
    return b->sink;
}
template <typename P>
__device__ __forceinline__ P *gp_check(const Bounds &b, P *p, unsigned bytes, unsigned site) {
    return (P *)bounds_check(&b, (const void *)p, bytes, site);
}
#define GPN(B, p, bytes) ::swab::gp_check((B), (p), (unsigned)(bytes), (kSwabFile << 16) | (unsigned)__LINE__)
#define GP(B, p) GPN(B, p, sizeof(*(p)))
#else
#define GPN(B, p, bytes) (p)
#define GP(B, p) (p)
#endif

// A wait gives up after this long (the kernels here run for micro- to
// milliseconds; a wait this long means a lost arrival).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------------------
// Geometry of one call.  Dilation is handled by residues: with stride s, the
// rows i = r + s*a (a = 0, 1, ...) of residue r only meet keys of the same
// residue, and on that subsequence the band is an undilated band with the
// same w and w_upper.  "sub-index" below means a.
// ---------------------------------------------------------------------------
struct Geom {
    int BH;       // b*h slices
    int n;        // sequence length
    int hd;       // head dim
    int w, wu;    // window left / right
    int s;        // key stride (dilation + 1)
    int D;        // band slots w + wu + 1
    int nsub;     // ceil(n / s): longest residue subsequence
    float padding;
    int h;                // heads: slice bh belongs to batch bh / h
    const float *kbias;   // [b, n] key-padding bias added to scaled scores, or null
    int drop_t;           // dropout threshold byte (0 = no dropout)
    unsigned long long seed;  // dropout key
    // Row strides (elements) of the dense tensors in the fused entry points:
    // 0 = contiguous [b, h, n, hd]; otherwise rows of [b, n, rs] with the heads
    // side by side (head hh at hh * hd).  rs_p: Q, K, V, dQ, dK, dV; rs_o: O, dO.
    long long rs_p, rs_o;
    // keep-bit cache of the fused dropout, or null: dm_nb words a query row
    uint32_t *dmask;
    int dm_nb;
#if SWAB_BOUNDS_CHECK
    Bounds bnd;   // the call's buffer extents (checked build)
#endif
};

// Element offset of dense row R = bh * n + i under row stride rs (R < 2^31:
// the descriptor check bounds b*h*n, so the divisions are 32-bit).
__host__ __device__ __forceinline__ long long dense_row(const Geom &g, long long R, long long rs) {
    if (rs == 0) return R * g.hd;
    const unsigned r = (unsigned)R, bh = r / (unsigned)g.n, i = r - bh * (unsigned)g.n;
    const unsigned b = bh / (unsigned)g.h, hh = bh - b * (unsigned)g.h;
    return ((long long)b * g.n + i) * rs + (long long)hh * g.hd;
}

__host__ __device__ __forceinline__ int residue_len(int n, int s, int r) {
    return r < n ? (n - r + s - 1) / s : 0;
}

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
template <typename T> struct Elt;
template <> struct Elt<float> {
    __device__ static __forceinline__ float to_f(float x) { return x; }
    __device__ static __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elt<__half> {
    __device__ static __forceinline__ float to_f(__half x) { return __half2float(x); }
    __device__ static __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct Elt<__nv_bfloat16> {
    __device__ static __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Two floats -> one 32-bit word of two 16-bit values (low = first), RNE.
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <typename T> __device__ __forceinline__ float lo16(uint32_t v);
template <typename T> __device__ __forceinline__ float hi16(uint32_t v);
template <> __device__ __forceinline__ float lo16<__half>(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
template <> __device__ __forceinline__ float hi16<__half>(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}
template <> __device__ __forceinline__ float lo16<__nv_bfloat16>(uint32_t v) {
    return __uint_as_float(v << 16);
}
template <> __device__ __forceinline__ float hi16<__nv_bfloat16>(uint32_t v) {
    return __uint_as_float(v & 0xffff0000u);
}

// ---------------------------------------------------------------------------
// misc PTX
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31) == 0; }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One arrival for a whole warp, made by lane 0 after a warp barrier that
// orders every lane's prior accesses before it: a barrier that warps signal
// this way counts warps, not threads (one shared-memory update per warp
// instead of one per thread).
__device__ __forceinline__ void mbar_arrive_warp(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with parity `parity` to complete.  Gives up
// (returns false) when `abort_flag` is raised by another thread, or after
// kWaitLimitNs, in which case it raises the flag and records a timeout in the
// device status word.  Never traps.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          volatile int *abort_flag, unsigned *err,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                if (err) atomicOr(err, kErrTimeout);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA: tiled tensor loads into shared memory, completing on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int x, int y, int z, int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
// Dense-tensor maps of the fused kernels are 4-D with increasing strides:
// {64, rows, h, b} for the contiguous layout, {64, h, rows, b} for rows of
// [b, n, rs]; `row` is the index within the map's residue.
__device__ __forceinline__ void tma_load_dense(void *dst, const CUtensorMap *map, uint64_t *bar,
                                               int row, int bh, int h, bool strided) {
    const int b = bh / h, hh = bh - b * h;
    if (strided) tma_load_4d(dst, map, bar, 0, hh, row, b);
    else tma_load_4d(dst, map, bar, 0, row, hh, b);
}
__device__ __forceinline__ void tma_prefetch_dense(const CUtensorMap *map, int row, int bh, int h,
                                                   bool strided) {
    const int b = bh / h, hh = bh - b * h;
    if (strided) tma_prefetch_l2_4d(map, 0, hh, row, b);
    else tma_prefetch_l2_4d(map, 0, row, hh, b);
}

// TMA reduce-add of a shared-memory tile into global memory (bulk group)
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, const void *src, int x, int y,
                                                  int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the source shared memory of every committed bulk group has been read
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed bulk group has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// bring a tile into L2 ahead of its load
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16 (fp32 accumulate):
// bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16,
// 1 = bf16), 15 / 16 A / B major (0 = K-major, 1 = MN-major), 17-22 N>>3,
// 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn, bool b_mn) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address >> 4
// (bits 0-13), leading byte offset >> 4 (16-29), stride byte offset >> 4
// (32-45), descriptor version 1 (bit 46), swizzle mode 2 = 128B (bits 61-63).
// K-major: rows of 128 B, SBO = 1024 between 8-row groups, LBO unused.
// MN-major: 128-B lines along MN, SBO = 1024 between 8-line K groups, LBO =
// distance between 64-element MN blocks.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A read from tensor memory (M rows = lanes,
// 16-bit elements packed two per 32-bit column along K)
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane
// (taddr.lane + t), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// Store 32 lanes x 32 consecutive 32-bit columns (the inverse of tmem_ld32).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// Store 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// TMEM address: lane in bits 31-16, column in bits 15-0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (sm_100 family): one instruction for two lanes of work
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 64x64->128 products with the
// published multipliers, the key bumped by the published Weyl constants
// between rounds.  The dropout keep byte of element (slice bh, query i, key j)
// is byte (b mod 32), b = floor(j / s), of the block at counter
// (floor(b / 32), i, bh, 0) and key (seed, 0), bytes little-endian from the
// four words.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x64_10(unsigned long long c0, unsigned long long c1,
                                              unsigned long long c2, unsigned long long c3,
                                              unsigned long long k0, unsigned long long k1,
                                              unsigned long long (&out)[4]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B97F4A7C15ull;
            k1 += 0xBB67AE8584CAA73Bull;
        }
        const unsigned long long hi0 = __umul64hi(0xD2E7470EE14C6C93ull, c0), lo0 = 0xD2E7470EE14C6C93ull * c0;
        const unsigned long long hi1 = __umul64hi(0xCA5A826395121157ull, c2), lo1 = 0xCA5A826395121157ull * c2;
        const unsigned long long n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// 32 keep bits of a block: bit k = (byte k >= t), bytes little-endian.
__device__ __forceinline__ uint32_t keep_bits32(const unsigned long long (&w)[4], int t) {
    const uint32_t t4 = 0x01010101u * (uint32_t)t;
    uint32_t bits = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t word = (uint32_t)(w[k >> 1] >> (32 * (k & 1)));
        const uint32_t ge = __vcmpgeu4(word, t4) & 0x01010101u;   // 1 per byte >= t
        bits |= ((ge * 0x01020408u) >> 24 & 0xFu) << (4 * k);      // bytes 4k..4k+3 -> bits
    }
    return bits;
}

// Transpose of a 32 x 32 bit matrix held by a warp, row `lane` in x (bit c =
// column c): returns column `lane` (bit r = row r).  Five butterfly steps;
// step j swaps, inside every 2j x 2j block, the upper right j x j block
// with the lower left one between the lanes j apart.
__device__ __forceinline__ uint32_t bit_transpose32(uint32_t x, int lane) {
    constexpr uint32_t kLeft[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int j = 16 >> k;
        const uint32_t m = kLeft[k];   // the columns c with (c & j) == 0
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) ? ((x & ~m) | ((y & ~m) >> j)) : ((x & m) | ((y & m) << j));
    }
    return x;
}

// Word of the keep-bit cache holding the keys [32 kb, 32 kb + 32) (sub-indices
// of the row's residue) of query position i, sub-index a: the row's words
// start at its first key block, floor(max(a - w, 0) / 32); -1 outside them.
__host__ __device__ __forceinline__ long long dmask_word(const Geom &g, long long bh, long long i, int a, int kb) {
    const int rel = kb - (a > g.w ? a - g.w : 0) / 32;
    if (rel < 0 || rel >= g.dm_nb) return -1;
    return (bh * g.n + i) * g.dm_nb + rel;
}

// keep-and-scale factor of one element (the exact fp32 paths)
__device__ __forceinline__ float drop_factor(const Geom &g, long long bh, long long i, long long j) {
    if (g.drop_t <= 0) return 1.f;
    const unsigned long long b = (unsigned long long)(j / g.s);
    unsigned long long w[4];
    philox4x64_10(b / 32, (unsigned long long)i, (unsigned long long)bh, 0, g.seed, 0, w);
    const int k = (int)(b % 32);
    const int byte = (int)((w[k >> 3] >> (8 * (k & 7))) & 0xffu);
    return byte >= g.drop_t ? 256.f / (256.f - (float)g.drop_t) : 0.f;
}

// fp32 add of 4 values into global memory (one vector reduction, sm_90+)
__device__ __forceinline__ void red_add4(float *dst, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// ---------------------------------------------------------------------------
// 16-byte global load / shared store helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void sts16(uint32_t saddr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

}  // namespace swab
