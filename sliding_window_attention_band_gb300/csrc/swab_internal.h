// swab_internal.h -- what the API translation unit (swab_api.cu) and the
// kernel translation units share: launch argument structs and the launchers.
// Each launcher enqueues its kernel(s) on `stream` and returns the launch's
// cudaError_t; validation has already been done by the caller.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "swab_common.cuh"

namespace swab {

// One 3-D tiled tensor map per residue r of the key stride: the rows
// r, r+s, r+2s, ... of every (b,h) slice of a [BH, n, 64] tensor, i.e.
// dims {64, ceil((n-r)/s), BH}, strides {s*64, n*64} elements.
struct TmapSet {
    CUtensorMap m[kMaxStride];
};

// Global-token description passed by value to kernels.
struct GlobArgs {
    int G;                 // number of global tokens (0 = none)
    int idx[kMaxGlobal];   // sorted positions
};

enum DType { kF32 = 0, kF16 = 1, kBF16 = 2 };

struct QKArgs {
    Geom g;
    float alpha;
    void *S;          // band output [BH, n, D]
    unsigned *err;    // device status word
    int nsplit;       // CTAs a query tile's key chunks are split over, one each (set by the launcher)
};

struct GatherArgs {
    Geom g;
    float alpha;
    const void *band; // band input [BH, n, D]
    void *out;        // dense output [BH, n, 64]
    unsigned *err;
    // global tokens (gl.G > 0 only)
    GlobArgs gl;
    const void *gw;   // band_pv: cols [BH, n, G]; band_t: rows [BH, G, n]
    const void *gy;   // the dense input whose G global rows enter (V or Y)
};

struct GlobScoreArgs {  // dense score pieces of band_qk
    Geom g;
    GlobArgs gl;
    float alpha;
    const void *A, *B;
    void *cols, *rows;
    unsigned *err;     // device status word (tensor-core kernel)
};

struct SoftmaxGlobArgs {
    Geom g;
    GlobArgs gl;
    const void *S, *S2;           // band inputs (fwd: S; bwd: P, dP)
    const void *Scols, *S2cols;   // cols inputs
    const void *Srows, *S2rows;   // rows inputs
    void *P, *Pcols, *Prows;      // outputs (fwd: P; bwd: dS)
    float *lse;
};

struct GlobReduceArgs {  // sums over the sequence for the G positions
    Geom g;
    GlobArgs gl;
    float alpha;
    const void *W;    // rows [BH, G, n] or cols [BH, n, G]
    const void *Y;    // [BH, n, 64]
    void *out;        // [BH, n, 64]; rows G[g] written / accumulated
};

struct DenseGlobArgs {  // fp32 band products with global tokens
    Geom g;
    GlobArgs gl;
    float alpha;
    const void *A, *B;
    const void *cols, *rows;
    void *out;
};

struct SoftmaxArgs {
    Geom g;
    const void *S;    // fwd: scores; bwd: P
    const void *S2;   // bwd: dP
    void *P;          // fwd: probabilities (may be null with Pd); bwd: dS
    float *lse;       // fwd only, may be null
    unsigned *err;
    void *Pd;         // fwd with dropout: dropped, rescaled probabilities; else null
};

struct AttnArgs {     // fused forward, tensor-core path
    Geom g;
    float scale;
    void *O;          // [BH, n, 64]
    float *lse;       // [BH, n] or null
    unsigned *err;
};

struct AttnArgsF32 {  // fused forward, fp32 path
    Geom g;
    float scale;
    const float *Q, *K, *V;
    float *O;
    float *lse;
};

struct BwdArgs {      // fused backward
    Geom g;
    float scale;
    const void *Q, *K, *V, *O, *dO;
    const float *lse;
    float *delta;     // workspace [BH, n]
    void *dQ, *dK, *dV;
    unsigned *err;
    float *dqacc;     // fused tensor-core path: fp32 dQ accumulator [BH, n, 64], or null
    // global tokens (fused tensor-core path with n_global > 0)
    int G;
    const void *gdK, *gdV;   // [BH, n, 64]: the global rows' dK, dV terms (every key)
    float *cdK, *cdV;        // [BH, G, 64] fp32: the global columns' dK (scaled), dV terms
};

struct DenseArgs {    // fp32 FFMA path
    Geom g;
    float alpha;
    const void *A;    // band_qk: A;  pv / t: band input
    const void *B;    // band_qk: B;  pv: V;  t: Y
    void *out;
};

// tensor-core paths (f16 / bf16, head_dim 64)
cudaError_t launch_band_qk_tc(DType dt, const TmapSet &mapA, const TmapSet &mapB,
                              const QKArgs &a, cudaStream_t st);
cudaError_t launch_band_gather_tc(DType dt, bool transposed, const TmapSet &mapB,
                                  const GatherArgs &a, cudaStream_t st);
size_t gather_glob_smem(int n, int G);      // extra shared memory with global tokens
size_t gather_smem_bytes(int n, int G);     // total shared memory of the gather kernel
// fused forward with global tokens: the band kernel with global keys masked,
// then the global columns merged into local rows and the global rows
cudaError_t launch_band_attention_glob(DType dt, const TmapSet &mapQ, const TmapSet &mapK,
                                       const TmapSet &mapV, const AttnArgs &a, const GlobArgs &gl,
                                       cudaStream_t st);
struct GlobalRowsArgs {   // dense rows of the global queries (fused forward)
    long long BH;
    int n;
    float scale;
    const void *Q, *K, *V;   // [BH, n, 64]
    void *O;                 // [BH, n, 64]: rows at the global positions written
    float *lse;              // [BH, n]
    GlobArgs gl;
    unsigned *err;           // device status word (tensor-core kernel)
    const float *kbias;      // [b, n] key-padding bias (natural-log units), or null
    int h;                   // heads: slice bh belongs to batch bh / h
#if SWAB_BOUNDS_CHECK
    Bounds bnd;              // the call's buffer extents (checked build)
#endif
};
// global columns on the tensor cores (G <= 64): map of Q (128-row boxes),
// contiguous [BH, n, 64]
cudaError_t launch_fused_glob_cols_tc(DType dt, const TmapSet &mq, const GlobalRowsArgs &a, cudaStream_t st);
// dense global rows on the tensor cores: maps of K, V (128-row boxes),
// contiguous [BH, n, 64]; f16/bf16
cudaError_t launch_fused_glob_rows_tc(DType dt, const TmapSet &mk, const TmapSet &mv, const GlobalRowsArgs &a,
                                      cudaStream_t st);
// cols_done / rows_done: the global columns were merged / the dense global
// rows written already (tensor-core kernels)
cudaError_t launch_fused_glob(DType dt, const Geom &g, const GlobArgs &gl, float scale, const void *Q,
                              const void *K, const void *V, void *O, float *lse, bool cols_done,
                              bool rows_done, cudaStream_t st);
cudaError_t launch_band_attention_tc(DType dt, const TmapSet &mapQ, const TmapSet &mapK,
                                     const TmapSet &mapV, const AttnArgs &a, cudaStream_t st);
cudaError_t launch_band_attention_f32(const AttnArgsF32 &a, cudaStream_t st);
cudaError_t launch_band_attention_bwd_tc(DType dt, const TmapSet &mq, const TmapSet &mk,
                                         const TmapSet &mv, const TmapSet &mo, const BwdArgs &a,
                                         cudaStream_t st);
cudaError_t launch_band_attention_bwd_f32(const BwdArgs &a, cudaStream_t st);
// one-pass backward (dK, dV and dQ in one persistent kernel; needs a.dqacc)
cudaError_t launch_band_attention_bwd_fused(DType dt, const TmapSet &mq, const TmapSet &mk,
                                            const TmapSet &mv, const TmapSet &mo, const TmapSet &macc,
                                            const BwdArgs &a, cudaStream_t st);
// SM count of the current device (swab_api.cu); 0 on error
int device_sm_count();
// dynamic shared-memory limit of a kernel, set once per (kernel, device) (swab_api.cu)
cudaError_t ensure_smem(const void *kernel, int bytes);
// the module-scope delta scratch of band_attention_bwd_noalloc (k_attention_bwd.cu);
// cudaErrorStreamCaptureUnsupported when the first lookup on a device would
// run while `st` is being captured
cudaError_t noalloc_delta_scratch(float **out, cudaStream_t st);
// fp32 FFMA paths
cudaError_t launch_band_qk_f32(const DenseArgs &a, cudaStream_t st);
cudaError_t launch_band_pv_f32(const DenseArgs &a, cudaStream_t st);
cudaError_t launch_band_t_f32(const DenseArgs &a, cudaStream_t st);
// global tokens
size_t glob_bitmap_bytes(int n);
cudaError_t launch_glob_scores(DType dt, const GlobScoreArgs &a, cudaStream_t st);
cudaError_t launch_softmax_glob(DType dt, const SoftmaxGlobArgs &a, bool bwd, cudaStream_t st);
// The vectorised softmax with global tokens (band rows of at most 32 values a
// lane; the dense global rows too when n is a multiple of a 16-byte piece and
// fits a CTA's registers).  Returns false, launching nothing, where it does
// not apply; *rows_done tells whether it also did the dense rows.
bool launch_softmax_glob_fast(DType dt, const SoftmaxGlobArgs &a, bool bwd, bool *rows_done,
                              cudaStream_t st, cudaError_t *err);
cudaError_t launch_glob_reduce(DType dt, const GlobReduceArgs &a, bool cols, cudaStream_t st);
// the same two on the tensor cores (f16 / bf16; k_global_tc.cu): maps of A, B
// (scores) or Y (reductions) over [BH, n, 64] with stride 1, 128- / 64-row boxes
cudaError_t launch_glob_scores_tc(DType dt, const TmapSet &mapA, const TmapSet &mapB, const GlobScoreArgs &a,
                                  cudaStream_t st);
cudaError_t launch_glob_reduce_tc(DType dt, const TmapSet &mapY, const GlobReduceArgs &a, bool cols, unsigned *err,
                                  cudaStream_t st);
cudaError_t launch_band_f32_glob(const DenseGlobArgs &a, bool transposed, cudaStream_t st);
// softmax forward / backward (all dtypes)
struct BiasTransposeArgs {   // AddBiasTranspose
    const void *X;     // rows of [b, n, M, h, hd]
    const void *bias;  // [M, h, hd] or null
    void *Y;           // [M, b, h, n, hd]
    long long rows;    // b * n
    long long b, n, h, M;
    long long cpr;     // 16-byte chunks per head row (hd * size / 16)
#if SWAB_BOUNDS_CHECK
    Bounds bnd;        // the call's buffer extents (checked build)
#endif
};
cudaError_t launch_add_bias_transpose(DType dt, const BiasTransposeArgs &a, cudaStream_t st);

struct GlobalProjArgs {   // global queries with their own projections
    long long BH;
    int G, n;
    float scale;
    const void *Qg;        // [BH, G, 64] compact global queries
    const void *Kg, *Vg;   // [BH, n, 64] global key / value projections
    void *Og;              // fwd: output [BH, G, 64]; bwd: the forward's output
    const void *dOg;       // bwd: [BH, G, 64]
    float *lseg;           // [BH, G]: fwd output (may be null), bwd input
    void *dQg, *dKg, *dVg; // bwd outputs
    float *ws;             // workspace (partials)
    int nchunks;           // set by the launcher
    unsigned *err;         // device status word (tensor-core backward)
    const float *kbias;    // [b, n] key-padding bias, or null (the fused backward's global rows)
    int h;                 // heads: slice bh belongs to batch bh / h
#if SWAB_BOUNDS_CHECK
    Bounds bnd;            // the call's buffer extents (checked build)
#endif
};
size_t global_proj_workspace_bytes(long long BH, int G, int n);
cudaError_t launch_global_proj(DType dt, const GlobalProjArgs &a, bool bwd, cudaStream_t st);
// tensor-core forward (f16 / bf16): maps of Kg, Vg (128-row boxes) and Qg (16-row boxes)
cudaError_t launch_global_proj_fwd_tc(DType dt, const TmapSet &mk, const TmapSet &mv, const TmapSet &mq,
                                      const GlobalProjArgs &a, cudaStream_t st);
// tensor-core backward (f16 / bf16): maps of Kg, Vg (128-row boxes) and of
// Qg, dOg (16-row boxes), one slice per third coordinate
cudaError_t launch_global_proj_bwd_tc(DType dt, const TmapSet &mk, const TmapSet &mv, const TmapSet &mq,
                                      const TmapSet &mo, const GlobalProjArgs &a, cudaStream_t st);
// the fused backward with global tokens (f16 / bf16, contiguous layout).  The
// workspace sections are set by the caller (swab_api.cu); maps:
//   band pass: mq, mk, mv, mo, macc as for launch_band_attention_bwd_fused;
//   global columns: mq1, mo1 (Q, dO with stride 1), mkc, mvc (the gathered
//   global keys / values, [BH, 128 ceil(G / 128), 64]), macc1 (the
//   accumulator, stride 1);
//   global rows: gp (Qg, Og, dOg, lseg, dQg, dKg = a.gdK, dVg = a.gdV, ws set)
//   with its maps gmk, gmv (K, V 128-row boxes), gmq, gmo (Qg, dOg 16-row boxes).
struct GlobBwdBufs {
    void *Qg, *Og, *dOg, *dQg;   // [BH, G, 64] gathered / the global rows' dQ
    float *lseg;                 // [BH, G]
    void *KG, *VG;               // [BH, 128 ceil(G / 128), 64]: the global keys, values, zero past G
};
cudaError_t launch_band_attention_bwd_glob(DType dt, const TmapSet &mq, const TmapSet &mk, const TmapSet &mv,
                                           const TmapSet &mo, const TmapSet &macc, const TmapSet &mq1,
                                           const TmapSet &mo1, const TmapSet &mkc, const TmapSet &mvc,
                                           const TmapSet &macc1, const GlobArgs &gl, const GlobBwdBufs &gb,
                                           const BwdArgs &a, const GlobalProjArgs &gp, const TmapSet &gmk,
                                           const TmapSet &gmv, const TmapSet &gmq, const TmapSet &gmo,
                                           cudaStream_t st);

cudaError_t launch_band_softmax(DType dt, const SoftmaxArgs &a, cudaStream_t st);
cudaError_t launch_band_softmax_bwd(DType dt, const SoftmaxArgs &a, cudaStream_t st);

// rows of one dense [BH, n, 64] tile box: band_qk loads 128-row boxes,
// the gather kernels 64-row boxes.
constexpr int kQKBoxRows = 128;
constexpr int kGatherBoxRows = 64;

}  // namespace swab
