// swab_api.cu -- the C ABI of include/swab.h: argument validation, tensor-map
// encoding, and kernel launches.  Validation runs on the host before any
// CUDA call, so a bad argument never reaches the GPU.  The library links the
// CUDA runtime statically and reaches the driver only through
// cudaGetDriverEntryPointByVersion, so it loads on a machine without a GPU.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>

#include "swab_internal.h"

static constexpr unsigned kSwabFile = 10;   // site id of the bounds checks

namespace swab {

// The device status word: bit k set = a kernel raised swab_status k.
__device__ unsigned g_status_word;

// Bounds-checked build: the first access a kernel found outside the call's
// extents (site + 1, address, bytes) and the scratch line such accesses are
// redirected to.  Present in both builds so the report reads zeros here.
__device__ unsigned long long g_bounds_rec[3];
__device__ __align__(256) unsigned char g_bounds_sink[256];

namespace {

// Self-test of the bounded wait every pipelined kernel uses: one warp waits on
// an mbarrier that nothing ever arrives at.  The wait must give up after
// `limit_ns`, record SWAB_ERR_TIMEOUT in the status word and return.
__global__ void k_selftest_wait(unsigned *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
    __syncthreads();
}

#if SWAB_BOUNDS_CHECK
// Self-test of the bounds checks: the extent handed in covers buf[0, 64);
// lane l stores to buf[l] (inside) and to buf[64 + l] (valid memory outside
// the extent), both through the check.
__device__ float g_selftest_buf[128];

__global__ void k_selftest_bounds(const Bounds b, float *buf) {
    const int l = threadIdx.x;
    *GP(b, buf + l) = (float)(l + 1);
    *GP(b, buf + 64 + l) = (float)(l + 1000);
}
#endif

const char *const kStatusNames[] = {
    "SWAB_OK", "SWAB_ERR_INVALID_ARG", "SWAB_ERR_UNSUPPORTED",
    "SWAB_ERR_MISALIGNED", "SWAB_ERR_CUDA", "SWAB_ERR_TIMEOUT", "SWAB_ERR_BOUNDS",
};

size_t elt_size(DType dt) { return dt == kF32 ? 4 : 2; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side checks of the descriptor; fills the kernel geometry.
swab_status check_desc(const swab_desc *d, Geom *g, DType *dt) {
    if (!d) return SWAB_ERR_INVALID_ARG;
    if (d->b < 1 || d->h < 1 || d->n < 1 || d->head_dim < 1) return SWAB_ERR_INVALID_ARG;
    if (d->w < 0 || d->w_upper < 0 || d->dilation < 0) return SWAB_ERR_INVALID_ARG;
    if (d->dtype != SWAB_F32 && d->dtype != SWAB_F16 && d->dtype != SWAB_BF16)
        return SWAB_ERR_INVALID_ARG;
    if (d->n_global < 0 || d->n_global > SWAB_MAX_GLOBAL) return SWAB_ERR_INVALID_ARG;
    if (d->n_global > 0) {
        if (!d->global_idx) return SWAB_ERR_INVALID_ARG;
        for (int k = 0; k < d->n_global; ++k) {
            const int32_t j = d->global_idx[k];
            if (j < 0 || j >= d->n) return SWAB_ERR_INVALID_ARG;
            if (k > 0 && d->global_idx[k - 1] >= j) return SWAB_ERR_INVALID_ARG;
        }
    }
    if (d->dilation > SWAB_MAX_DILATION) return SWAB_ERR_UNSUPPORTED;
    if (d->key_bias && reinterpret_cast<uintptr_t>(d->key_bias) % 4 != 0) return SWAB_ERR_MISALIGNED;
    if (!(d->dropout_p >= 0.f && d->dropout_p < 1.f)) return SWAB_ERR_INVALID_ARG;  // NaN too
    const int drop_t = (int)std::min(255.f, std::nearbyint(d->dropout_p * 256.f));
    if (drop_t > 0 && d->n_global > 0) return SWAB_ERR_UNSUPPORTED;  // dropout with globals
    const long long BH = (long long)d->b * d->h;
    const long long D = (long long)d->w + d->w_upper + 1;
    if (BH > 65535) return SWAB_ERR_UNSUPPORTED;          // grid z
    if (D > (1ll << 24)) return SWAB_ERR_UNSUPPORTED;
    if (BH * d->n > 0x7fffffffll) return SWAB_ERR_UNSUPPORTED;  // row index fits int32 grid
    if (d->dtype == SWAB_F32) {
        if (d->head_dim > 128) return SWAB_ERR_UNSUPPORTED;
    } else if (d->head_dim != 64) {
        return SWAB_ERR_UNSUPPORTED;
    }
    g->BH = (int)BH;
    g->n = d->n;
    g->hd = d->head_dim;
    g->w = d->w;
    g->wu = d->w_upper;
    g->s = d->dilation + 1;
    g->D = (int)D;
    g->nsub = (d->n + g->s - 1) / g->s;
    g->padding = d->padding;
    g->h = d->h;
    g->kbias = d->key_bias;
    g->drop_t = drop_t;
    g->seed = d->dropout_seed;
    // strided dense layout: rows of [b, n, rs] (heads side by side); the TMA
    // maps need 16-byte row strides
    const long long hw = (long long)d->h * d->head_dim;
    const long long vec = 16 / (long long)elt_size(static_cast<DType>(d->dtype));
    for (const int64_t rs : {d->qkv_row_stride, d->out_row_stride}) {
        if (rs < 0 || (rs > 0 && rs < hw)) return SWAB_ERR_INVALID_ARG;
        if (rs % vec != 0) return SWAB_ERR_MISALIGNED;
        if (rs > 0 && (long long)d->n * rs * vec > (1ll << 40)) return SWAB_ERR_UNSUPPORTED;
    }
    g->rs_p = d->qkv_row_stride;
    g->rs_o = d->out_row_stride;
    // the keep-bit cache: used by the fused calls with dropout only
    g->dmask = drop_t > 0 ? d->dropout_mask : nullptr;
    g->dm_nb = (int)((D + 31) / 32 + 1);
    if (g->dmask && reinterpret_cast<uintptr_t>(g->dmask) % 4 != 0) return SWAB_ERR_MISALIGNED;
    *dt = static_cast<DType>(d->dtype);
    return SWAB_OK;
}

swab_status check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs) {
        if (!p) return SWAB_ERR_INVALID_ARG;
        if (!aligned16(p)) return SWAB_ERR_MISALIGNED;
    }
    return SWAB_OK;
}

// ---------------------------------------------------------------------------
// driver entry point for tensor-map encoding
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

#if SWAB_BOUNDS_CHECK
bool map_fits(const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides, size_t es);
#endif

// One map per residue r: rows r, r+s, ... of every slice of a [BH, n, 64]
// tensor; box = 64 elements x box_rows rows, 128-byte swizzle, zero fill
// outside the residue's rows.
bool build_rows_maps(TmapSet *set, const void *base, const Geom &g, DType dt, int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    const size_t es = elt_size(dt);
    const CUtensorMapDataType ty =
        dt == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    std::memset(set, 0, sizeof(*set));
    for (int r = 0; r < g.s; ++r) {
        int nr = residue_len(g.n, g.s, r);
        const int rr = nr > 0 ? r : 0;  // empty residue: never loaded, encode a valid map
        if (nr == 0) nr = 1;
        cuuint64_t dims[3] = {64, (cuuint64_t)nr, (cuuint64_t)g.BH};
        cuuint64_t strides[2] = {(cuuint64_t)g.s * 64 * es, (cuuint64_t)g.n * 64 * es};
        cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        void *ptr = const_cast<char *>(static_cast<const char *>(base)) + (size_t)rr * 64 * es;
#if SWAB_BOUNDS_CHECK
        if (!map_fits(ptr, 3, dims, strides, es)) return false;
#endif
        CUresult res = enc(&set->m[r], ty, 3, ptr, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (res != CUDA_SUCCESS) return false;
    }
    return true;
}

// Maps of the fused kernels' dense tensors, one per residue r: 4-D with
// increasing strides (TMA coordinates in tma_load_dense).  rs == 0: the
// contiguous [b, h, n, 64] layout as {64, rows, h, b}; rs > 0: rows of
// [b, n, rs] with head hh at column 64 hh, as {64, h, rows, b}.  Box = 64
// elements x box_rows rows of one (b, h) slice, 128-byte swizzle.
bool build_dense_maps(TmapSet *set, const void *base, const Geom &g, DType dt, int box_rows,
                      long long rs) {
    auto enc = get_encode();
    if (!enc) return false;
    const size_t es = elt_size(dt);
    const CUtensorMapDataType ty =
        dt == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int b = g.BH / g.h;
    std::memset(set, 0, sizeof(*set));
    for (int r = 0; r < g.s; ++r) {
        int nr = residue_len(g.n, g.s, r);
        const int rr = nr > 0 ? r : 0;  // empty residue: never loaded, encode a valid map
        if (nr == 0) nr = 1;
        cuuint64_t dims[4], strides[3];
        cuuint32_t box[4];
        size_t first;
        if (rs == 0) {
            dims[0] = 64; dims[1] = (cuuint64_t)nr; dims[2] = (cuuint64_t)g.h; dims[3] = (cuuint64_t)b;
            strides[0] = (cuuint64_t)g.s * 64 * es;
            strides[1] = (cuuint64_t)g.n * 64 * es;
            strides[2] = (cuuint64_t)g.h * g.n * 64 * es;
            box[0] = 64; box[1] = (cuuint32_t)box_rows; box[2] = 1; box[3] = 1;
            first = (size_t)rr * 64 * es;
        } else {
            dims[0] = 64; dims[1] = (cuuint64_t)g.h; dims[2] = (cuuint64_t)nr; dims[3] = (cuuint64_t)b;
            strides[0] = 64 * es;
            strides[1] = (cuuint64_t)g.s * rs * es;
            strides[2] = (cuuint64_t)g.n * rs * es;
            box[0] = 64; box[1] = 1; box[2] = (cuuint32_t)box_rows; box[3] = 1;
            first = (size_t)rr * rs * es;
        }
        cuuint32_t estr[4] = {1, 1, 1, 1};
        void *ptr = const_cast<char *>(static_cast<const char *>(base)) + first;
#if SWAB_BOUNDS_CHECK
        if (!map_fits(ptr, 4, dims, strides, es)) return false;
#endif
        CUresult res = enc(&set->m[r], ty, 4, ptr, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (res != CUDA_SUCCESS) return false;
    }
    return true;
}

// One map per residue r over an fp32 [BH, n, 64] accumulator: box = 32 floats
// (128 B) x 128 rows, 128-byte swizzle; the one-pass backward adds its dQ
// tiles into it with TMA reduce-add stores.
bool build_acc_maps(TmapSet *set, float *base, const Geom &g) {
    auto enc = get_encode();
    if (!enc) return false;
    std::memset(set, 0, sizeof(*set));
    for (int r = 0; r < g.s; ++r) {
        int nr = residue_len(g.n, g.s, r);
        const int rr = nr > 0 ? r : 0;
        if (nr == 0) nr = 1;
        cuuint64_t dims[3] = {64, (cuuint64_t)nr, (cuuint64_t)g.BH};
        cuuint64_t strides[2] = {(cuuint64_t)g.s * 64 * 4, (cuuint64_t)g.n * 64 * 4};
        cuuint32_t box[3] = {32, 128, 1};
        cuuint32_t estr[3] = {1, 1, 1};
#if SWAB_BOUNDS_CHECK
        if (!map_fits(base + (size_t)rr * 64, 3, dims, strides, 4)) return false;
#endif
        CUresult res = enc(&set->m[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base + (size_t)rr * 64, dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (res != CUDA_SUCCESS) return false;
    }
    return true;
}

// Address of the status word on the current device (cached per device).
unsigned *status_word() {
    static std::mutex mu;
    static unsigned *cache[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned *>(p);
    }
    return cache[dev];
}

// ---------------------------------------------------------------------------
// Extents of a call's buffers (bounds-checked build).  Each entry point lists
// its buffers with the byte sizes the descriptor gives them; the list goes
// into the kernels' arguments and, for the tensor maps' footprints, into a
// thread-local copy.  In the regular build SWAB_BOUNDS is SWAB_OK.
// ---------------------------------------------------------------------------
struct Extent {
    const void *p;
    size_t bytes;
};

size_t round16(size_t bytes) { return (bytes + 15) / 16 * 16; }

// Byte sizes of a call's buffers as the descriptor lays them out.
size_t bh_n(const swab_desc *d) { return (size_t)d->b * d->h * d->n; }
size_t esize(const swab_desc *d) { return d->dtype == SWAB_F32 ? 4 : 2; }
// dense [b, h, n, hd], or rows of [b, n, rs] with this head block the last
size_t dense_bytes(const swab_desc *d, long long rs) {
    if (rs == 0) return bh_n(d) * d->head_dim * esize(d);
    return ((size_t)d->b * d->n - 1) * (size_t)rs * esize(d) + (size_t)d->h * d->head_dim * esize(d);
}
// band [b, h, n, D], readable to the next 16-byte boundary
size_t band_bytes(const swab_desc *d) {
    return round16(bh_n(d) * ((size_t)d->w + d->w_upper + 1) * esize(d));
}
size_t glob_bytes(const swab_desc *d) { return bh_n(d) * (size_t)d->n_global * esize(d); }
size_t rows_f32_bytes(const swab_desc *d) { return bh_n(d) * 4; }
size_t kbias_bytes(const swab_desc *d) { return (size_t)d->b * d->n * 4; }
// the companions of band tensors (null entries are skipped)
Extent gcols(const swab_desc *d, const swab_glob *q) { return {d->n_global > 0 && q ? q->cols : nullptr, glob_bytes(d)}; }
Extent grows(const swab_desc *d, const swab_glob *q) { return {d->n_global > 0 && q ? q->rows : nullptr, glob_bytes(d)}; }

#if SWAB_BOUNDS_CHECK
thread_local Bounds t_bounds;        // the current call's extents
thread_local bool t_map_overhang;    // one of its tensor maps overhung them

swab_status set_bounds(Bounds *b, std::initializer_list<Extent> ext) {
    t_map_overhang = false;
    Bounds nb{};
    for (const Extent &e : ext) {
        if (!e.p || e.bytes == 0) continue;
        if (nb.n == kBoundsMax) return SWAB_ERR_UNSUPPORTED;
        nb.lo[nb.n] = reinterpret_cast<unsigned long long>(e.p);
        nb.hi[nb.n] = nb.lo[nb.n] + e.bytes;
        ++nb.n;
    }
    void *rec = nullptr, *sink = nullptr;
    if (cudaGetSymbolAddress(&rec, g_bounds_rec) != cudaSuccess ||
        cudaGetSymbolAddress(&sink, g_bounds_sink) != cudaSuccess)
        return SWAB_ERR_CUDA;
    nb.err = status_word();
    if (!nb.err) return SWAB_ERR_CUDA;
    nb.rec = static_cast<unsigned long long *>(rec);
    nb.sink = sink;
    *b = nb;
    t_bounds = nb;
    return SWAB_OK;
}

// The bytes a tensor map can address, [base, base + (dims[0]-1) es +
// sum_k (dims[k]-1) strides[k-1] + es), lie inside one extent of the call.
bool map_fits(const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides, size_t es) {
    unsigned long long last = (dims[0] - 1) * es;
    for (int k = 1; k < rank; ++k) last += (dims[k] - 1) * strides[k - 1];
    const unsigned long long lo = reinterpret_cast<unsigned long long>(base), hi = lo + last + es;
    for (int k = 0; k < t_bounds.n; ++k)
        if (lo >= t_bounds.lo[k] && hi <= t_bounds.hi[k]) return true;
    t_map_overhang = true;
    return false;
}
#define SWAB_BOUNDS(target, ...) ::swab::set_bounds((target), {__VA_ARGS__})
#else
#define SWAB_BOUNDS(target, ...) SWAB_OK
#endif

// The status of a failed CUDA step: SWAB_ERR_BOUNDS when a tensor map of the
// call overhung its extents (checked build), else SWAB_ERR_CUDA.
swab_status fail_cuda() {
#if SWAB_BOUNDS_CHECK
    if (t_map_overhang) return SWAB_ERR_BOUNDS;
#endif
    return SWAB_ERR_CUDA;
}

swab_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SWAB_OK : fail_cuda(); }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Global tokens: companion tensors must be given, head_dim must be 64 and the
// kernels' shared-memory bitmap (n bits) plus the G dense rows must fit.
swab_status check_globals(const swab_desc *d, std::initializer_list<const swab_glob *> globs,
                          GlobArgs *gl) {
    gl->G = d->n_global;
    if (d->n_global == 0) return SWAB_OK;
    if (d->head_dim != 64) return SWAB_ERR_UNSUPPORTED;
    if (gather_smem_bytes(d->n, d->n_global) > 227 * 1024) return SWAB_ERR_UNSUPPORTED;
    for (const swab_glob *q : globs) {
        if (!q || !q->cols || !q->rows) return SWAB_ERR_INVALID_ARG;
        if (!aligned16(q->cols) || !aligned16(q->rows)) return SWAB_ERR_MISALIGNED;
    }
    for (int k = 0; k < d->n_global; ++k) gl->idx[k] = d->global_idx[k];
    return SWAB_OK;
}

swab_status check_no_globals(const swab_desc *d) {
    return d->n_global > 0 ? SWAB_ERR_UNSUPPORTED : SWAB_OK;
}

// The sums over the sequence for the G global outputs: tensor cores for f16 /
// bf16 (the dense operand Y in 64-row boxes, stride 1), exact FFMA for fp32.
cudaError_t glob_reduce(DType dt, const GlobReduceArgs &r, bool cols, cudaStream_t st) {
    if (dt == kF32) return launch_glob_reduce(dt, r, cols, st);
    Geom g1 = r.g;
    g1.s = 1;
    g1.nsub = r.g.n;
    TmapSet my;
    if (!build_rows_maps(&my, r.Y, g1, dt, 64)) return cudaErrorInvalidValue;
    unsigned *err = status_word();
    if (!err) return cudaErrorInvalidValue;
    return launch_glob_reduce_tc(dt, my, r, cols, err, st);
}

// The two transposed-product names share this body.
swab_status band_t_common(const swab_desc *desc, float alpha, const void *Bd, const swab_glob *Bg,
                          const void *Y, void *X, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if (g.rs_p || g.rs_o) return SWAB_ERR_UNSUPPORTED;  // dense tensors contiguous here
    GlobArgs gl;
    if ((s = check_globals(desc, {Bg}, &gl)) != SWAB_OK) return s;
    if ((s = check_ptrs({Bd, Y, X})) != SWAB_OK) return s;
    if ((s = SWAB_BOUNDS(&g.bnd, {Bd, band_bytes(desc)}, gcols(desc, Bg), grows(desc, Bg), {Y, dense_bytes(desc, 0)},
                         {X, dense_bytes(desc, 0)})) != SWAB_OK)
        return s;
    cudaStream_t st = as_stream(stream);
    cudaError_t e;
    if (dt == kF32) {
        if (gl.G > 0) {
            DenseGlobArgs a{g, gl, alpha, Bd, Y, Bg->cols, Bg->rows, X};
            e = launch_band_f32_glob(a, true, st);
        } else {
            DenseArgs a{g, alpha, Bd, Y, X};
            e = launch_band_t_f32(a, st);
        }
    } else {
        TmapSet mapY;
        if (!build_rows_maps(&mapY, Y, g, dt, kGatherBoxRows)) return fail_cuda();
        unsigned *err = status_word();
        if (!err) return fail_cuda();
        GatherArgs a{g, alpha, Bd, X, err, gl, gl.G > 0 ? Bg->rows : nullptr, Y};
        e = launch_band_gather_tc(dt, true, mapY, a, st);
    }
    if (e == cudaSuccess && gl.G > 0) {
        GlobReduceArgs r{g, gl, alpha, Bg->cols, Y, X};
        e = glob_reduce(dt, r, true, st);
    }
    return from_cuda(e);
}

}  // namespace

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`; cudaFuncSetAttribute runs only when the limit recorded for
// (kernel, device) is lower, so repeated launches (and stream capture) skip it.
cudaError_t ensure_smem(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    int &have = done[std::make_pair(kernel, dev)];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

// Number of SMs of the current device (cached per device); 0 on error.
int device_sm_count() {
    static std::mutex mu;
    static int cache[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = v;
    }
    return cache[dev];
}

}  // namespace swab

using namespace swab;

extern "C" {

SWAB_API const char *swab_version(void) { return "0.1.0"; }

SWAB_API const char *swab_status_string(swab_status status) {
    const int k = static_cast<int>(status);
    if (k < 0 || k >= (int)(sizeof(kStatusNames) / sizeof(kStatusNames[0])))
        return "SWAB_UNKNOWN_STATUS";
    return kStatusNames[k];
}

SWAB_API swab_status swab_selftest_wait_timeout(uint32_t limit_us, void *stream) {
    if (limit_us == 0 || limit_us > 1000000u) return SWAB_ERR_INVALID_ARG;
    unsigned *err = status_word();
    if (!err) return fail_cuda();
    k_selftest_wait<<<1, 32, 0, as_stream(stream)>>>(err, 1000ull * limit_us);
    return from_cuda(cudaGetLastError());
}

SWAB_API int32_t swab_bounds_checked(void) { return SWAB_BOUNDS_CHECK ? 1 : 0; }

SWAB_API swab_status swab_bounds_report(uint64_t *out, int32_t reset) {
    if (!out) return SWAB_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return SWAB_ERR_CUDA;
    unsigned long long rec[3] = {0, 0, 0};
    if (cudaMemcpyFromSymbol(rec, g_bounds_rec, sizeof(rec)) != cudaSuccess) return SWAB_ERR_CUDA;
    for (int k = 0; k < 3; ++k) out[k] = rec[k];
    if (reset) {
        const unsigned long long zero[3] = {0, 0, 0};
        if (cudaMemcpyToSymbol(g_bounds_rec, zero, sizeof(zero)) != cudaSuccess) return SWAB_ERR_CUDA;
    }
    return SWAB_OK;
}

SWAB_API swab_status swab_selftest_bounds(void *stream) {
#if SWAB_BOUNDS_CHECK
    void *buf = nullptr;
    if (cudaGetSymbolAddress(&buf, g_selftest_buf) != cudaSuccess) return SWAB_ERR_CUDA;
    Bounds b;
    const swab_status s = set_bounds(&b, {{buf, 64 * sizeof(float)}});
    if (s != SWAB_OK) return s;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(buf, 0, 128 * sizeof(float), st) != cudaSuccess) return SWAB_ERR_CUDA;
    k_selftest_bounds<<<1, 32, 0, st>>>(b, static_cast<float *>(buf));
    if (cudaGetLastError() != cudaSuccess) return SWAB_ERR_CUDA;
    float host[128];
    if (cudaMemcpyAsync(host, buf, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SWAB_ERR_CUDA;
    // the stores inside the extent landed, the ones outside it did not
    for (int l = 0; l < 32; ++l)
        if (host[l] != (float)(l + 1) || host[64 + l] != 0.f) return SWAB_ERR_BOUNDS;
    return SWAB_OK;
#else
    (void)stream;
    return SWAB_ERR_UNSUPPORTED;
#endif
}

SWAB_API swab_status swab_device_status(int32_t *flags, int32_t reset) {
    if (!flags) return SWAB_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return fail_cuda();
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return fail_cuda();
    *flags = static_cast<int32_t>(v);
    if (reset) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
            return fail_cuda();
    }
    return SWAB_OK;
}

SWAB_API swab_status band_qk(const swab_desc *desc, float alpha, const void *A, const void *B,
                             void *S, const swab_glob *Sg, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if (g.rs_p || g.rs_o) return SWAB_ERR_UNSUPPORTED;  // dense tensors contiguous here
    GlobArgs gl;
    if ((s = check_globals(desc, {Sg}, &gl)) != SWAB_OK) return s;
    if ((s = check_ptrs({A, B, S})) != SWAB_OK) return s;
    if ((s = SWAB_BOUNDS(&g.bnd, {A, dense_bytes(desc, 0)}, {B, dense_bytes(desc, 0)}, {S, band_bytes(desc)},
                         gcols(desc, Sg), grows(desc, Sg))) != SWAB_OK)
        return s;
    cudaStream_t st = as_stream(stream);
    cudaError_t e;
    if (dt == kF32) {
        DenseArgs a{g, alpha, A, B, S};
        e = launch_band_qk_f32(a, st);
    } else {
        TmapSet mapA, mapB;
        if (!build_rows_maps(&mapA, A, g, dt, kQKBoxRows) ||
            !build_rows_maps(&mapB, B, g, dt, kQKBoxRows))
            return fail_cuda();
        unsigned *err = status_word();
        if (!err) return fail_cuda();
        QKArgs a{g, alpha, S, err};
        e = launch_band_qk_tc(dt, mapA, mapB, a, st);
    }
    if (e == cudaSuccess && gl.G > 0) {
        GlobScoreArgs a{g, gl, alpha, A, B, Sg->cols, Sg->rows};
        if (dt == kF32) {
            e = launch_glob_scores(dt, a, st);
        } else {
            // tensor cores: 128-row tiles of A and B in sequence order
            Geom g1 = g;
            g1.s = 1;
            g1.nsub = g.n;
            TmapSet ma, mb;
            if (!build_rows_maps(&ma, A, g1, dt, 128) || !build_rows_maps(&mb, B, g1, dt, 128)) return fail_cuda();
            a.err = status_word();
            if (!a.err) return fail_cuda();
            e = launch_glob_scores_tc(dt, ma, mb, a, st);
        }
    }
    return from_cuda(e);
}

SWAB_API swab_status band_softmax(const swab_desc *desc, const void *S, const swab_glob *Sg,
                                  void *P, const swab_glob *Pg, float *lse, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if (g.drop_t > 0) return SWAB_ERR_UNSUPPORTED;  // the dropped output: band_softmax_dropout
    GlobArgs gl;
    if ((s = check_globals(desc, {Sg, Pg}, &gl)) != SWAB_OK) return s;
    if ((s = check_ptrs({S, P})) != SWAB_OK) return s;
    if (lse && !aligned16(lse)) return SWAB_ERR_MISALIGNED;
    if ((s = SWAB_BOUNDS(&g.bnd, {S, band_bytes(desc)}, {P, band_bytes(desc)}, gcols(desc, Sg), grows(desc, Sg),
                         gcols(desc, Pg), grows(desc, Pg), {lse, rows_f32_bytes(desc)},
                         {g.kbias, kbias_bytes(desc)})) != SWAB_OK)
        return s;
    if (gl.G > 0) {
        SoftmaxGlobArgs a{g, gl, S, nullptr, Sg->cols, nullptr, Sg->rows, nullptr,
                          P, Pg->cols, Pg->rows, lse};
        return from_cuda(launch_softmax_glob(dt, a, false, as_stream(stream)));
    }
    SoftmaxArgs a{g, S, nullptr, P, lse, nullptr};
    return from_cuda(launch_band_softmax(dt, a, as_stream(stream)));
}

SWAB_API swab_status add_bias_transpose(const swab_desc *desc, int32_t M, const void *X,
                                        const void *bias, void *Y, void *stream) {
    if (!desc || M < 1) return SWAB_ERR_INVALID_ARG;
    if (desc->b < 1 || desc->h < 1 || desc->n < 1 || desc->head_dim < 1) return SWAB_ERR_INVALID_ARG;
    if (desc->dtype != SWAB_F32 && desc->dtype != SWAB_F16 && desc->dtype != SWAB_BF16)
        return SWAB_ERR_INVALID_ARG;
    const DType dt = static_cast<DType>(desc->dtype);
    const long long row_bytes = (long long)desc->head_dim * (long long)elt_size(dt);
    if (row_bytes % 16 != 0) return SWAB_ERR_UNSUPPORTED;
    swab_status s;
    if ((s = check_ptrs({X, Y})) != SWAB_OK) return s;
    if (bias && !aligned16(bias)) return SWAB_ERR_MISALIGNED;
    BiasTransposeArgs a{X, bias, Y, (long long)desc->b * desc->n, desc->b, desc->n, desc->h, M,
                        row_bytes / 16};
    const long long total = a.rows * a.M * a.h * row_bytes;
    if (a.rows > 0x7fffffffLL || a.M * a.h * a.cpr > (1LL << 30)) return SWAB_ERR_UNSUPPORTED;
    if (total / row_bytes / a.rows / a.M != a.h) return SWAB_ERR_UNSUPPORTED;  // overflow
    // Y must not overlap X
    const char *x0 = static_cast<const char *>(X), *y0 = static_cast<const char *>(Y);
    if (x0 < y0 + total && y0 < x0 + total) return SWAB_ERR_INVALID_ARG;
    if ((s = SWAB_BOUNDS(&a.bnd, {X, (size_t)total}, {bias, (size_t)(a.M * a.h * row_bytes)}, {Y, (size_t)total})) !=
        SWAB_OK)
        return s;
    return from_cuda(launch_add_bias_transpose(dt, a, as_stream(stream)));
}

// shared checks of the global-query calls; fills the kernel arguments
static swab_status global_proj_setup(const swab_desc *desc, float scale, GlobalProjArgs *a,
                                     DType *dt) {
    Geom g;
    swab_status s = check_desc(desc, &g, dt);
    if (s != SWAB_OK) return s;
    if (desc->n_global < 1) return SWAB_ERR_INVALID_ARG;
    if (desc->head_dim != 64) return SWAB_ERR_UNSUPPORTED;
    if (g.rs_p || g.rs_o) return SWAB_ERR_UNSUPPORTED;
    if (g.kbias) return SWAB_ERR_UNSUPPORTED;   // no key bias in the separate projections
    *a = GlobalProjArgs{};
    a->BH = g.BH;
    a->G = desc->n_global;
    a->n = g.n;
    a->scale = scale;
    return SWAB_OK;
}

SWAB_API size_t global_attention_workspace(const swab_desc *desc) {
    if (!desc || desc->b < 1 || desc->h < 1 || desc->n < 1 || desc->n_global < 1) return 0;
    return global_proj_workspace_bytes((long long)desc->b * desc->h, desc->n_global, desc->n);
}

SWAB_API swab_status global_attention(const swab_desc *desc, float scale, const void *Qg,
                                      const void *Kg, const void *Vg, void *Og, float *lseg,
                                      void *workspace, void *stream) {
    GlobalProjArgs a;
    DType dt;
    swab_status s = global_proj_setup(desc, scale, &a, &dt);
    if (s != SWAB_OK) return s;
    if ((s = check_ptrs({Qg, Kg, Vg, Og, workspace})) != SWAB_OK) return s;
    if (lseg && !aligned16(lseg)) return SWAB_ERR_MISALIGNED;
    a.Qg = Qg;
    a.Kg = Kg;
    a.Vg = Vg;
    a.Og = Og;
    a.lseg = lseg;
    a.ws = static_cast<float *>(workspace);
    {
        const size_t gq = (size_t)a.BH * a.G * 64 * elt_size(dt), kv = (size_t)a.BH * a.n * 64 * elt_size(dt);
        if ((s = SWAB_BOUNDS(&a.bnd, {Qg, gq}, {Kg, kv}, {Vg, kv}, {Og, gq}, {lseg, (size_t)a.BH * a.G * 4},
                             {workspace, global_attention_workspace(desc)})) != SWAB_OK)
            return s;
    }
    if (dt == kF32) return from_cuda(launch_global_proj(dt, a, false, as_stream(stream)));
    Geom gk{}, gq{};
    gk.BH = gq.BH = (int)a.BH;
    gk.s = gq.s = 1;
    gk.n = a.n;
    gq.n = a.G;
    TmapSet mk, mv, mq;
    if (!build_rows_maps(&mk, Kg, gk, dt, 128) || !build_rows_maps(&mv, Vg, gk, dt, 128) ||
        !build_rows_maps(&mq, Qg, gq, dt, 16))
        return fail_cuda();
    a.err = status_word();
    if (!a.err) return fail_cuda();
    return from_cuda(launch_global_proj_fwd_tc(dt, mk, mv, mq, a, as_stream(stream)));
}

SWAB_API swab_status global_attention_bwd(const swab_desc *desc, float scale, const void *Qg,
                                          const void *Kg, const void *Vg, const void *Og,
                                          const void *dOg, const float *lseg, void *dQg,
                                          void *dKg, void *dVg, void *workspace, void *stream) {
    GlobalProjArgs a;
    DType dt;
    swab_status s = global_proj_setup(desc, scale, &a, &dt);
    if (s != SWAB_OK) return s;
    if ((s = check_ptrs({Qg, Kg, Vg, Og, dOg, lseg, dQg, dKg, dVg, workspace})) != SWAB_OK) return s;
    a.Qg = Qg;
    a.Kg = Kg;
    a.Vg = Vg;
    a.Og = const_cast<void *>(Og);
    a.dOg = dOg;
    a.lseg = const_cast<float *>(lseg);
    a.dQg = dQg;
    a.dKg = dKg;
    a.dVg = dVg;
    a.ws = static_cast<float *>(workspace);
    {
        const size_t gq = (size_t)a.BH * a.G * 64 * elt_size(dt), kv = (size_t)a.BH * a.n * 64 * elt_size(dt);
        if ((s = SWAB_BOUNDS(&a.bnd, {Qg, gq}, {Kg, kv}, {Vg, kv}, {Og, gq}, {dOg, gq}, {lseg, (size_t)a.BH * a.G * 4},
                             {dQg, gq}, {dKg, kv}, {dVg, kv}, {workspace, global_attention_workspace(desc)})) != SWAB_OK)
            return s;
    }
    if (dt == kF32) return from_cuda(launch_global_proj(dt, a, true, as_stream(stream)));
    // tensor-core path: [n, 64] slices of Kg, Vg and [G, 64] slices of Qg, dOg
    Geom gk{}, gq{};
    gk.BH = gq.BH = (int)a.BH;
    gk.s = gq.s = 1;
    gk.n = a.n;
    gq.n = a.G;
    TmapSet mk, mv, mq, mo;
    if (!build_rows_maps(&mk, Kg, gk, dt, 128) || !build_rows_maps(&mv, Vg, gk, dt, 128) ||
        !build_rows_maps(&mq, Qg, gq, dt, 16) || !build_rows_maps(&mo, dOg, gq, dt, 16))
        return fail_cuda();
    a.err = status_word();
    if (!a.err) return fail_cuda();
    return from_cuda(launch_global_proj_bwd_tc(dt, mk, mv, mq, mo, a, as_stream(stream)));
}

// Largest band the softmax kernels take with dropout: the per-row keep bits
// (one word per 32 keys, four rows per block) stay within 32 KB of shared memory.
constexpr int kMaxDropBand = 65536;

SWAB_API swab_status band_softmax_dropout(const swab_desc *desc, const void *S, void *P, void *Pd,
                                          float *lse, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if (desc->n_global > 0) return SWAB_ERR_UNSUPPORTED;
    if ((s = check_ptrs({S, Pd})) != SWAB_OK) return s;
    if (P && !aligned16(P)) return SWAB_ERR_MISALIGNED;
    if (lse && !aligned16(lse)) return SWAB_ERR_MISALIGNED;
    if (g.D > kMaxDropBand) return SWAB_ERR_UNSUPPORTED;
    if ((s = SWAB_BOUNDS(&g.bnd, {S, band_bytes(desc)}, {P, band_bytes(desc)}, {Pd, band_bytes(desc)},
                         {lse, rows_f32_bytes(desc)}, {g.kbias, kbias_bytes(desc)})) != SWAB_OK)
        return s;
    SoftmaxArgs a{g, S, nullptr, P, lse, nullptr, Pd};
    return from_cuda(launch_band_softmax(dt, a, as_stream(stream)));
}

SWAB_API swab_status band_pv(const swab_desc *desc, float alpha, const void *P,
                             const swab_glob *Pg, const void *V, void *O, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if (g.rs_p || g.rs_o) return SWAB_ERR_UNSUPPORTED;  // dense tensors contiguous here
    GlobArgs gl;
    if ((s = check_globals(desc, {Pg}, &gl)) != SWAB_OK) return s;
    if ((s = check_ptrs({P, V, O})) != SWAB_OK) return s;
    if ((s = SWAB_BOUNDS(&g.bnd, {P, band_bytes(desc)}, gcols(desc, Pg), grows(desc, Pg), {V, dense_bytes(desc, 0)},
                         {O, dense_bytes(desc, 0)})) != SWAB_OK)
        return s;
    cudaStream_t st = as_stream(stream);
    cudaError_t e;
    if (dt == kF32) {
        if (gl.G > 0) {
            DenseGlobArgs a{g, gl, alpha, P, V, Pg->cols, Pg->rows, O};
            e = launch_band_f32_glob(a, false, st);
        } else {
            DenseArgs a{g, alpha, P, V, O};
            e = launch_band_pv_f32(a, st);
        }
    } else {
        TmapSet mapV;
        if (!build_rows_maps(&mapV, V, g, dt, kGatherBoxRows)) return fail_cuda();
        unsigned *err = status_word();
        if (!err) return fail_cuda();
        GatherArgs a{g, alpha, P, O, err, gl, gl.G > 0 ? Pg->cols : nullptr, V};
        e = launch_band_gather_tc(dt, false, mapV, a, st);
    }
    if (e == cudaSuccess && gl.G > 0) {
        GlobReduceArgs r{g, gl, alpha, Pg->rows, V, O};
        e = glob_reduce(dt, r, false, st);
    }
    return from_cuda(e);
}

SWAB_API swab_status band_qk_bwd_t(const swab_desc *desc, float alpha, const void *dS,
                                   const swab_glob *dSg, const void *Q, void *dK, void *stream) {
    return band_t_common(desc, alpha, dS, dSg, Q, dK, stream);
}

SWAB_API swab_status band_pv_bwd_t(const swab_desc *desc, float alpha, const void *P,
                                   const swab_glob *Pg, const void *dO, void *dV, void *stream) {
    return band_t_common(desc, alpha, P, Pg, dO, dV, stream);
}

SWAB_API swab_status band_softmax_bwd(const swab_desc *desc, const void *P, const swab_glob *Pg,
                                      const void *dP, const swab_glob *dPg, void *dS,
                                      const swab_glob *dSg, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    GlobArgs gl;
    if ((s = check_globals(desc, {Pg, dPg, dSg}, &gl)) != SWAB_OK) return s;
    if ((s = check_ptrs({P, dP, dS})) != SWAB_OK) return s;
    if (g.drop_t > 0 && g.D > kMaxDropBand) return SWAB_ERR_UNSUPPORTED;
    if ((s = SWAB_BOUNDS(&g.bnd, {P, band_bytes(desc)}, {dP, band_bytes(desc)}, {dS, band_bytes(desc)}, gcols(desc, Pg),
                         grows(desc, Pg), gcols(desc, dPg), grows(desc, dPg), gcols(desc, dSg),
                         grows(desc, dSg))) != SWAB_OK)
        return s;
    if (gl.G > 0) {
        SoftmaxGlobArgs a{g, gl, P, dP, Pg->cols, dPg->cols, Pg->rows, dPg->rows,
                          dS, dSg->cols, dSg->rows, nullptr};
        return from_cuda(launch_softmax_glob(dt, a, true, as_stream(stream)));
    }
    SoftmaxArgs a{g, P, dP, dS, nullptr, nullptr};
    return from_cuda(launch_band_softmax_bwd(dt, a, as_stream(stream)));
}

SWAB_API swab_status band_attention(const swab_desc *desc, float scale, const void *Q,
                                    const void *K, const void *V, void *O, float *lse,
                                    void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if ((s = check_ptrs({Q, K, V, O})) != SWAB_OK) return s;
    if (lse && !aligned16(lse)) return SWAB_ERR_MISALIGNED;
    if ((s = SWAB_BOUNDS(&g.bnd, {Q, dense_bytes(desc, g.rs_p)}, {K, dense_bytes(desc, g.rs_p)},
                         {V, dense_bytes(desc, g.rs_p)}, {O, dense_bytes(desc, g.rs_o)}, {lse, rows_f32_bytes(desc)},
                         {g.kbias, kbias_bytes(desc)},
                         {g.dmask, g.dmask ? band_attention_dropout_mask_bytes(desc) : 0})) != SWAB_OK)
        return s;
    if (desc->n_global > 0) {
        // band keys outside G by the fused kernel, then the global columns
        // merged into local rows (needs lse) and the global rows
        if (dt == kF32 || g.rs_p || g.rs_o) return SWAB_ERR_UNSUPPORTED;
        if (!lse) return SWAB_ERR_INVALID_ARG;
        if ((long long)(g.n + 31) / 32 * 4 > 23 * 1024) return SWAB_ERR_UNSUPPORTED;   // key bitmap
        GlobArgs gl;
        gl.G = desc->n_global;
        for (int k = 0; k < gl.G; ++k) gl.idx[k] = desc->global_idx[k];
        TmapSet mq, mk, mv;
        if (!build_dense_maps(&mq, Q, g, dt, kQKBoxRows, 0) || !build_dense_maps(&mk, K, g, dt, kQKBoxRows, 0) ||
            !build_dense_maps(&mv, V, g, dt, kQKBoxRows, 0))
            return fail_cuda();
        unsigned *err = status_word();
        if (!err) return fail_cuda();
        AttnArgs a{g, scale, O, lse, err};
        cudaStream_t st = as_stream(stream);
        cudaError_t e = launch_band_attention_glob(dt, mq, mk, mv, a, gl, st);
        Geom gr{};   // rows of [BH, n, 64] in 128-row boxes
        gr.BH = g.BH;
        gr.n = g.n;
        gr.s = 1;
        GlobalRowsArgs r{g.BH, g.n, scale, Q, K, V, O, lse, gl, err, g.kbias, g.h};
#if SWAB_BOUNDS_CHECK
        r.bnd = g.bnd;
#endif
        bool cols_done = false, rows_done = false;
        if (e == cudaSuccess && gl.G <= 64) {
            // the global columns on the tensor cores
            TmapSet mq1;
            if (!build_rows_maps(&mq1, Q, gr, dt, 128)) return fail_cuda();
            e = launch_fused_glob_cols_tc(dt, mq1, r, st);
            cols_done = true;
        }
        const int sms = device_sm_count();
        if (e == cudaSuccess && sms > 0 && 2LL * ((gl.G + 15) / 16) * g.BH >= sms) {
            // the dense global rows on the tensor cores, when their (16-query
            // chunk, slice) CTAs fill the GPU
            TmapSet mk1, mv1;
            if (!build_rows_maps(&mk1, K, gr, dt, 128) || !build_rows_maps(&mv1, V, gr, dt, 128))
                return fail_cuda();
            e = launch_fused_glob_rows_tc(dt, mk1, mv1, r, st);
            rows_done = true;
        }
        if (e == cudaSuccess) e = launch_fused_glob(dt, g, gl, scale, Q, K, V, O, lse, cols_done, rows_done, st);
        return from_cuda(e);
    }
    if (dt == kF32) {
        AttnArgsF32 a{g, scale, static_cast<const float *>(Q), static_cast<const float *>(K),
                      static_cast<const float *>(V), static_cast<float *>(O), lse};
        return from_cuda(launch_band_attention_f32(a, as_stream(stream)));
    }
    TmapSet mq, mk, mv;
    if (!build_dense_maps(&mq, Q, g, dt, kQKBoxRows, g.rs_p) ||
        !build_dense_maps(&mk, K, g, dt, kQKBoxRows, g.rs_p) ||
        !build_dense_maps(&mv, V, g, dt, kQKBoxRows, g.rs_p))
        return fail_cuda();
    unsigned *err = status_word();
    if (!err) return fail_cuda();
    AttnArgs a{g, scale, O, lse, err};
    return from_cuda(launch_band_attention_tc(dt, mq, mk, mv, a, as_stream(stream)));
}

// Workspace of band_attention_bwd with global tokens, after the per-row delta
// and the fp32 dQ accumulator: byte offsets of each section (256-aligned).
struct BwdGlobLayout {
    size_t Qg, Og, dOg, dQg, lseg, KG, VG, gdK, gdV, cdK, cdV, gp, end;
};
static size_t up256(size_t x) { return (x + 255) / 256 * 256; }
static BwdGlobLayout bwd_glob_layout(const swab_desc *desc, size_t start) {
    const size_t BH = (size_t)desc->b * desc->h, n = desc->n, G = desc->n_global, es = 2;
    BwdGlobLayout L;
    size_t o = up256(start);
    auto take = [&](size_t bytes) { const size_t at = o; o = up256(o + bytes); return at; };
    L.Qg = take(BH * G * 64 * es);
    L.Og = take(BH * G * 64 * es);
    L.dOg = take(BH * G * 64 * es);
    L.dQg = take(BH * G * 64 * es);
    L.lseg = take(BH * G * 4);
    const size_t grows = (G + 127) / 128 * 128;   // whole 128-key tiles of gathered global keys
    L.KG = take(BH * grows * 64 * es);
    L.VG = take(BH * grows * 64 * es);
    L.gdK = take(BH * n * 64 * es);
    L.gdV = take(BH * n * 64 * es);
    L.cdK = take(BH * G * 64 * 4);
    L.cdV = take(BH * G * 64 * 4);
    L.gp = take(global_proj_workspace_bytes((long long)BH, (int)G, (int)n));
    L.end = o;
    return L;
}

SWAB_API size_t band_attention_dropout_mask_bytes(const swab_desc *desc) {
    if (!desc || desc->b < 1 || desc->h < 1 || desc->n < 1 || desc->w < 0 || desc->w_upper < 0) return 0;
    const size_t D = (size_t)desc->w + desc->w_upper + 1;
    return (size_t)desc->b * desc->h * desc->n * ((D + 31) / 32 + 1) * sizeof(uint32_t);
}

SWAB_API size_t band_attention_bwd_workspace(const swab_desc *desc) {
    if (!desc || desc->b < 1 || desc->h < 1 || desc->n < 1) return 0;
    const size_t rows = (size_t)desc->b * desc->h * desc->n;
    const size_t delta = (rows * sizeof(float) + 255) / 256 * 256;
    if (desc->dtype == SWAB_F32) return delta;
    // fp16 / bf16: the per-row delta, then the fp32 dQ accumulator [rows, 64]
    const size_t base = delta + rows * 64 * sizeof(float);
    if (desc->n_global > 0 && desc->n_global <= SWAB_MAX_GLOBAL) return bwd_glob_layout(desc, base).end;
    return base;
}

// band_attention_bwd with global tokens (f16 / bf16, contiguous layout, no key
// bias or dropout): the band pass with global keys and queries left out, the
// global columns as a pass of the same kernel over the gathered global keys,
// and the global rows through the global-query backward (the shared Q, K, V
// are their projections); all scratch in the caller's workspace.
static swab_status bwd_with_globals(const swab_desc *desc, const Geom &g, DType dt, BwdArgs a, cudaStream_t st) {
    GlobArgs gl;
    swab_status s = check_globals(desc, {}, &gl);
    if (s != SWAB_OK) return s;
    if (dt == kF32 || g.rs_p || g.rs_o || g.drop_t > 0) return SWAB_ERR_UNSUPPORTED;
    if ((long long)(g.n + 31) / 32 * 4 > 12 * 1024) return SWAB_ERR_UNSUPPORTED;   // key bitmap in shared memory
    const size_t rows = (size_t)g.BH * g.n;
    char *ws = static_cast<char *>(static_cast<void *>(a.delta));
    a.dqacc = reinterpret_cast<float *>(ws + up256(rows * sizeof(float)));
    const BwdGlobLayout L = bwd_glob_layout(desc, up256(rows * sizeof(float)) + rows * 64 * sizeof(float));
    GlobBwdBufs gb;
    gb.Qg = ws + L.Qg;
    gb.Og = ws + L.Og;
    gb.dOg = ws + L.dOg;
    gb.dQg = ws + L.dQg;
    gb.lseg = reinterpret_cast<float *>(ws + L.lseg);
    gb.KG = ws + L.KG;
    gb.VG = ws + L.VG;
    a.G = gl.G;
    a.gdK = ws + L.gdK;
    a.gdV = ws + L.gdV;
    a.cdK = reinterpret_cast<float *>(ws + L.cdK);
    a.cdV = reinterpret_cast<float *>(ws + L.cdV);
    a.err = status_word();
    if (!a.err) return fail_cuda();
    // band pass: the per-residue maps
    TmapSet mq, mk, mv, mo, macc;
    if (!build_dense_maps(&mq, a.Q, g, dt, kQKBoxRows, 0) || !build_dense_maps(&mk, a.K, g, dt, kQKBoxRows, 0) ||
        !build_dense_maps(&mv, a.V, g, dt, kQKBoxRows, 0) || !build_dense_maps(&mo, a.dO, g, dt, kQKBoxRows, 0) ||
        !build_acc_maps(&macc, a.dqacc, g))
        return fail_cuda();
    // global columns: Q, dO and the accumulator with stride 1; the gathered
    // global keys / values as [b, h, 128 x ceil(G / 128), 64]
    Geom g1 = g;
    g1.s = 1;
    g1.nsub = g.n;
    Geom gk = g;
    gk.s = 1;
    gk.n = (gl.G + 127) / 128 * 128;
    gk.nsub = gk.n;
    TmapSet mq1, mo1, mkc, mvc, macc1;
    if (!build_dense_maps(&mq1, a.Q, g1, dt, kQKBoxRows, 0) || !build_dense_maps(&mo1, a.dO, g1, dt, kQKBoxRows, 0) ||
        !build_dense_maps(&mkc, gb.KG, gk, dt, kQKBoxRows, 0) || !build_dense_maps(&mvc, gb.VG, gk, dt, kQKBoxRows, 0) ||
        !build_acc_maps(&macc1, a.dqacc, g1))
        return fail_cuda();
    // global rows: the global-query backward with Kg = K, Vg = V
    GlobalProjArgs gp{};
    gp.BH = g.BH;
    gp.G = gl.G;
    gp.n = g.n;
    gp.scale = a.scale;
    gp.Qg = gb.Qg;
    gp.Kg = a.K;
    gp.Vg = a.V;
    gp.Og = gb.Og;
    gp.dOg = gb.dOg;
    gp.lseg = gb.lseg;
    gp.dQg = gb.dQg;
    gp.dKg = const_cast<void *>(a.gdK);
    gp.dVg = const_cast<void *>(a.gdV);
    gp.ws = reinterpret_cast<float *>(ws + L.gp);
    gp.err = a.err;
    gp.kbias = g.kbias;   // the global rows see the key bias of every key
    gp.h = g.h;
#if SWAB_BOUNDS_CHECK
    gp.bnd = g.bnd;
#endif
    Geom gkr{}, gqr{};
    gkr.BH = gqr.BH = g.BH;
    gkr.s = gqr.s = 1;
    gkr.n = g.n;
    gqr.n = gl.G;
    TmapSet gmk, gmv, gmq, gmo;
    if (!build_rows_maps(&gmk, a.K, gkr, dt, 128) || !build_rows_maps(&gmv, a.V, gkr, dt, 128) ||
        !build_rows_maps(&gmq, gb.Qg, gqr, dt, 16) || !build_rows_maps(&gmo, gb.dOg, gqr, dt, 16))
        return fail_cuda();
    return from_cuda(launch_band_attention_bwd_glob(dt, mq, mk, mv, mo, macc, mq1, mo1, mkc, mvc, macc1, gl, gb, a,
                                                    gp, gmk, gmv, gmq, gmo, st));
}

SWAB_API swab_status band_attention_bwd(const swab_desc *desc, float scale, const void *Q,
                                        const void *K, const void *V, const void *O,
                                        const void *dO, const float *lse, void *dQ, void *dK,
                                        void *dV, void *workspace, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if ((s = check_ptrs({Q, K, V, O, dO, lse, dQ, dK, dV, workspace})) != SWAB_OK) return s;
    if ((s = SWAB_BOUNDS(&g.bnd, {Q, dense_bytes(desc, g.rs_p)}, {K, dense_bytes(desc, g.rs_p)},
                         {V, dense_bytes(desc, g.rs_p)}, {O, dense_bytes(desc, g.rs_o)}, {dO, dense_bytes(desc, g.rs_o)},
                         {lse, rows_f32_bytes(desc)}, {dQ, dense_bytes(desc, g.rs_p)}, {dK, dense_bytes(desc, g.rs_p)},
                         {dV, dense_bytes(desc, g.rs_p)}, {workspace, band_attention_bwd_workspace(desc)},
                         {g.kbias, kbias_bytes(desc)},
                         {g.dmask, g.dmask ? band_attention_dropout_mask_bytes(desc) : 0})) != SWAB_OK)
        return s;
    cudaStream_t st = as_stream(stream);
    BwdArgs a{g, scale, Q, K, V, O, dO, lse, static_cast<float *>(workspace), dQ, dK, dV, nullptr};
    if (desc->n_global > 0) return bwd_with_globals(desc, g, dt, a, st);
    if (dt == kF32) return from_cuda(launch_band_attention_bwd_f32(a, st));
    TmapSet mq, mk, mv, mo;
    if (!build_dense_maps(&mq, Q, g, dt, kQKBoxRows, g.rs_p) ||
        !build_dense_maps(&mk, K, g, dt, kQKBoxRows, g.rs_p) ||
        !build_dense_maps(&mv, V, g, dt, kQKBoxRows, g.rs_p) ||
        !build_dense_maps(&mo, dO, g, dt, kQKBoxRows, g.rs_o))
        return fail_cuda();
    a.err = status_word();
    if (!a.err) return fail_cuda();
    const size_t rows = (size_t)g.BH * g.n;
    a.dqacc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                        (rows * sizeof(float) + 255) / 256 * 256);
    TmapSet macc;
    if (!build_acc_maps(&macc, a.dqacc, g)) return fail_cuda();
    return from_cuda(launch_band_attention_bwd_fused(dt, mq, mk, mv, mo, macc, a, st));
}

SWAB_API swab_status band_attention_bwd_noalloc(const swab_desc *desc, float scale, const void *Q,
                                                const void *K, const void *V, const void *O,
                                                const void *dO, const float *lse, void *dQ,
                                                void *dK, void *dV, void *stream) {
    Geom g;
    DType dt;
    swab_status s = check_desc(desc, &g, &dt);
    if (s != SWAB_OK) return s;
    if ((s = check_no_globals(desc)) != SWAB_OK) return s;
    if ((long long)g.BH * g.n > (long long)SWAB_NOALLOC_MAX_ROWS) return SWAB_ERR_UNSUPPORTED;
    if (desc->key_bias) return SWAB_ERR_UNSUPPORTED;  // the two-kernel path has no key bias
    if (g.drop_t > 0) return SWAB_ERR_UNSUPPORTED;    // nor dropout
    if (g.rs_p || g.rs_o) return SWAB_ERR_UNSUPPORTED;  // nor the strided layout
    if ((s = check_ptrs({Q, K, V, O, dO, lse, dQ, dK, dV})) != SWAB_OK) return s;
    cudaStream_t st = as_stream(stream);
    float *scratch = nullptr;
    const cudaError_t se = noalloc_delta_scratch(&scratch, st);
    if (se == cudaErrorStreamCaptureUnsupported) return SWAB_ERR_UNSUPPORTED;
    if (se != cudaSuccess) return fail_cuda();
    if ((s = SWAB_BOUNDS(&g.bnd, {Q, dense_bytes(desc, 0)}, {K, dense_bytes(desc, 0)}, {V, dense_bytes(desc, 0)},
                         {O, dense_bytes(desc, 0)}, {dO, dense_bytes(desc, 0)}, {lse, rows_f32_bytes(desc)},
                         {dQ, dense_bytes(desc, 0)}, {dK, dense_bytes(desc, 0)}, {dV, dense_bytes(desc, 0)},
                         {scratch, (size_t)SWAB_NOALLOC_MAX_ROWS * sizeof(float)})) != SWAB_OK)
        return s;
    BwdArgs a{g, scale, Q, K, V, O, dO, lse, scratch, dQ, dK, dV, nullptr};
    if (dt == kF32) return from_cuda(launch_band_attention_bwd_f32(a, st));
    TmapSet mq, mk, mv, mo;
    if (!build_rows_maps(&mq, Q, g, dt, kQKBoxRows) || !build_rows_maps(&mk, K, g, dt, kQKBoxRows) ||
        !build_rows_maps(&mv, V, g, dt, kQKBoxRows) || !build_rows_maps(&mo, dO, g, dt, kQKBoxRows))
        return fail_cuda();
    a.err = status_word();
    if (!a.err) return fail_cuda();
    return from_cuda(launch_band_attention_bwd_tc(dt, mq, mk, mv, mo, a, st));
}

}  // extern "C"
