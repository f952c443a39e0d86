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
};

struct GatherArgs {
    Geom g;
    float alpha;
    const void *band; // band input [BH, n, D]
    void *out;        // dense output [BH, n, 64]
    unsigned *err;
};

struct SoftmaxArgs {
    Geom g;
    const void *S;    // fwd: scores; bwd: P
    const void *S2;   // bwd: dP
    void *P;          // fwd: probabilities; bwd: dS
    float *lse;       // fwd only, may be null
    unsigned *err;
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
cudaError_t launch_band_attention_tc(DType dt, const TmapSet &mapQ, const TmapSet &mapK,
                                     const TmapSet &mapV, const AttnArgs &a, cudaStream_t st);
cudaError_t launch_band_attention_f32(const AttnArgsF32 &a, cudaStream_t st);
// fp32 FFMA paths
cudaError_t launch_band_qk_f32(const DenseArgs &a, cudaStream_t st);
cudaError_t launch_band_pv_f32(const DenseArgs &a, cudaStream_t st);
cudaError_t launch_band_t_f32(const DenseArgs &a, cudaStream_t st);
// softmax forward / backward (all dtypes)
cudaError_t launch_band_softmax(DType dt, const SoftmaxArgs &a, cudaStream_t st);
cudaError_t launch_band_softmax_bwd(DType dt, const SoftmaxArgs &a, cudaStream_t st);

// rows of one dense [BH, n, 64] tile box: band_qk loads 128-row boxes,
// the gather kernels 64-row boxes.
constexpr int kQKBoxRows = 128;
constexpr int kGatherBoxRows = 64;

}  // namespace swab
