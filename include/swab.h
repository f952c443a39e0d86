/*
 * swab.h -- C ABI of the sliding-window (banded) attention library for one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (pages: "Developing a faster schedule for Longformer's
 * kernel", TVM forum, posts 1, 3, 5 and 6):
 *   Longformer attention is built from a banded ("diagonal") matrix product:
 *   of Q.K^T only the diagonals k in [-w, w_upper] are computed, with
 *   dilation d (key stride s = d + 1), so query row i meets key
 *       j = i + k*s,   k = t - w,   slot t in [0, D),   D = w + w_upper + 1.
 *   A slot whose key falls outside [0, n) holds the constant `padding`.
 *   Post 6 names three modes of one kernel: the forward product (dense x
 *   dense^T -> band, t3d3 = 2w+1) and two backward products (band x dense,
 *   transpose_t1 = 0, and band^T x dense, transpose_t1 = 1).  The author
 *   merged them into one function only because they could not put several
 *   kernels into one .so; here they are separate entry points.
 *
 * Global tokens ("[WIP] Improve LongformerAttention performance", ONNX
 * Runtime issue, item (1): one global index of length S shared by the batch):
 *   G sorted, unique positions shared by every (b, h).  A row i not in G
 *   attends to its band keys that are not in G plus all of G; a row in G
 *   attends to every key.  The extra dense pieces live in caller-owned
 *   companion tensors (swab_glob): `cols` [b,h,n,G] holds every row's value
 *   at the G global keys, `rows` [b,h,G,n] holds the dense rows of the G
 *   global queries.  Band slots whose key is in G, and the band rows and
 *   `cols` rows of global queries, are not used by attention.
 *
 * Conventions for every entry point:
 *   - Layouts are row-major and contiguous: dense tensors (Q, K, V, O, dO,
 *     dQ, dK, dV) [b,h,n,head_dim]; band tensors (S, P, dP, dS) [b,h,n,D];
 *     lse [b,h,n] fp32.  Element type = desc->dtype for all but lse.
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned.  Band tensors must be readable up to the next 16-byte
 *     boundary past their last element (any cudaMalloc / PyTorch allocation
 *     is).  The library allocates, frees and synchronises nothing.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it; results are ready when the stream reaches them.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed validation returns an error and launches nothing.
 *   - Invalid slots (key outside [0, n)) of an INPUT band tensor are ignored,
 *     whatever they hold; `padding` is written only by band_qk.
 *   - No entry point aborts or prints.  A launch failure returns
 *     SWAB_ERR_CUDA.  Device-side waits are bounded: a wait that gives up
 *     records SWAB_ERR_TIMEOUT in the library's device status word, read with
 *     swab_device_status().
 *   - Tensor-core paths: dtype f16/bf16 with head_dim 64.  dtype f32 runs an
 *     exact-fp32 FFMA path (head_dim 1..128).
 */
#ifndef SWAB_H
#define SWAB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define SWAB_API __declspec(dllexport)
#else
#define SWAB_API __attribute__((visibility("default")))
#endif

#define SWAB_MAX_GLOBAL 256  /* most global tokens per call */
#define SWAB_MAX_DILATION 15 /* key stride at most 16 */
#define SWAB_NOALLOC_MAX_ROWS (1u << 22) /* b*h*n limit of band_attention_bwd_noalloc */

typedef enum swab_status {
    SWAB_OK = 0,
    SWAB_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad global index */
    SWAB_ERR_UNSUPPORTED = 2, /* head_dim / dtype / size outside what is built */
    SWAB_ERR_MISALIGNED = 3,  /* a tensor pointer is not 16-byte aligned */
    SWAB_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed */
    SWAB_ERR_TIMEOUT = 5,     /* a device wait gave up (see swab_device_status) */
    SWAB_ERR_BOUNDS = 6       /* bounds-checked build only: a kernel's global access
                                 fell outside the call's buffers (swab_bounds_report) */
} swab_status;

typedef enum swab_dtype { SWAB_F32 = 0, SWAB_F16 = 1, SWAB_BF16 = 2 } swab_dtype;

/* Problem description: the kernel parameters of the TVM forum thread, posts
 * 5-6 (b, n, h, w, w_upper, padding; the head dimension replaces m = 768
 * divided over h = 12 heads) plus the dilation of post 3 and the global
 * index of the ONNX Runtime issue. */
typedef struct swab_desc {
    int32_t b;                 /* batch */
    int32_t h;                 /* heads (merged with the batch: slices b*h) */
    int32_t n;                 /* sequence length, >= 1 */
    int32_t head_dim;          /* 64 for f16/bf16; 1..128 for f32 */
    int32_t w;                 /* keys on the left, >= 0 */
    int32_t w_upper;           /* keys on the right, >= 0 (0 = autoregressive) */
    int32_t dilation;          /* 0..SWAB_MAX_DILATION; key stride dilation+1 */
    float padding;             /* value band_qk writes where the key is outside [0,n) */
    int32_t dtype;             /* swab_dtype of every tensor except lse */
    int32_t n_global;          /* G, 0..SWAB_MAX_GLOBAL; 0 = no global tokens */
    const int32_t *global_idx; /* HOST array of G sorted unique positions in [0,n) */
    /* Optional key-padding bias (nvFuser issue "HuggingFace BertForMaskedLM -
     * Log Softmax Fusion...", fusion 1, adds (1 - mask) * -10000 per key to the
     * scaled scores): DEVICE array of b*n fp32, 4-byte aligned, row bb holding
     * the term added to the score of every query of batch bb with key j
     * before the softmax; NULL for none.  Read by band_softmax, band_attention
     * and band_attention_bwd (the other calls do not depend on it).  With
     * n_global > 0 the fused pair adds it to every key a row attends to: the
     * band keys and the global columns of a local row, every key of a global
     * row; band_softmax likewise adds it to the band slots, the global
     * columns (key global_idx[g]) and the dense global rows.
     * global_attention, global_attention_bwd and band_attention_bwd_noalloc
     * return SWAB_ERR_UNSUPPORTED when it is set. */
    const float *key_bias;
    /* Optional dropout of the attention probabilities (the nvFuser fusion 1
     * dropout, p with 1/(1-p) scaling), in band_attention and
     * band_attention_bwd (pass the same values to both): dropout_p in [0, 1) is
     * rounded to t = round(256 * dropout_p) (at most 255); an element is kept
     * with probability 1 - t/256 and then scaled by 256 / (256 - t).  Element
     * (slice bh, query i, key j) is kept iff byte (b mod 32), b = floor(j / s),
     * of the Philox4x64-10 block at counter (floor(b / 32), i, bh, 0) and key
     * (dropout_seed, 0) -- bytes little-endian from the four output words --
     * is >= t.  lse is that of the probabilities before dropout.  Read by
     * band_softmax_dropout, band_softmax_bwd, band_attention and
     * band_attention_bwd; with t > 0, band_softmax (use band_softmax_dropout),
     * global tokens and band_attention_bwd_noalloc return SWAB_ERR_UNSUPPORTED;
     * the other calls do not depend on it. */
    float dropout_p;
    uint64_t dropout_seed;
    /* Optional strided layout of the dense tensors in band_attention and
     * band_attention_bwd (ONNX Runtime issue "[WIP] Improve LongformerAttention
     * performance": the merged QKV projection leaves rows of [b, n, 3, h,
     * head_dim]).  0 = the contiguous [b, h, n, head_dim] layout.  Otherwise
     * the row stride in elements: element (batch bb, head hh, position i,
     * channel c) is at (bb * n + i) * stride + hh * head_dim + c, i.e. rows of
     * [b, n, stride] with the heads side by side; stride >= h * head_dim and a
     * multiple of 16 bytes (else SWAB_ERR_INVALID_ARG / SWAB_ERR_MISALIGNED).
     * qkv_row_stride applies to Q, K, V, dQ, dK, dV (3 h head_dim reads Q, K, V
     * straight from the merged projection: pass its base, base + h head_dim and
     * base + 2 h head_dim); out_row_stride to O and dO.  lse stays [b, h, n].
     * The other calls (materialised band products, band_attention_bwd_noalloc)
     * take the contiguous layout only (SWAB_ERR_UNSUPPORTED). */
    int64_t qkv_row_stride;
    int64_t out_row_stride;
    /* Optional keep-bit cache of the fused dropout (f16 / bf16 band_attention
     * and band_attention_bwd with dropout_p > 0): DEVICE buffer of
     * band_attention_dropout_mask_bytes(desc) bytes, 4-byte aligned; NULL for
     * none.  band_attention writes into it the keep bits it draws (32 keys of
     * a query row to a word); band_attention_bwd, given the buffer that
     * band_attention filled for the same description (sizes, window, dilation,
     * dropout_p, dropout_seed), reads them instead of drawing them again.  The
     * decisions are the same either way.  The other calls ignore it. */
    uint32_t *dropout_mask;
} swab_desc;

/* Companion of a band tensor when n_global > 0 (device pointers, dtype of the
 * band tensor).  Pass NULL when n_global == 0. */
typedef struct swab_glob {
    void *cols; /* [b,h,n,G]: value of row i at key global_idx[g] */
    void *rows; /* [b,h,G,n]: dense row of query global_idx[g] over all keys */
} swab_glob;

/* Forward product (TVM thread, post 6: dense x dense^T -> t3d3 = D diagonals):
 *   S[i,t] = alpha * sum_c A[i,c] * B[j,c]  with j = i + (t-w)*s in [0,n),
 *   S[i,t] = padding otherwise; accumulation in fp32, one round-to-nearest
 *   into the output dtype.
 * Forward scores: A = Q, B = K, alpha = 1/sqrt(head_dim).  Backward:
 * A = dO, B = V, alpha = 1 gives dP.  With globals, also writes
 * Sg->cols[i,g] = alpha*A[i].B[G[g]] and Sg->rows[g,j] = alpha*A[G[g]].B[j]. */
SWAB_API swab_status band_qk(const swab_desc *desc, float alpha, const void *A, const void *B,
                             void *S, const swab_glob *Sg, void *stream);

/* Masked row softmax over the band (nvFuser issue "HuggingFace
 * BertForMaskedLM - Log Softmax Fusion...", fusion 1: max, exp(x - max), sum,
 * divide, in fp32):
 *   P[i,t] = exp(S[i,t] - m_i) / Z_i on used slots, 0 on the others;
 *   lse[i] = m_i + log Z_i (lse may be NULL).
 * With globals the row also covers Sg->cols (written to Pg->cols); a global
 * query's row is the dense Sg->rows row (written to Pg->rows) and its band
 * row and cols row are written as zeros. */
SWAB_API swab_status band_softmax(const swab_desc *desc, const void *S, const swab_glob *Sg,
                                  void *P, const swab_glob *Pg, float *lse, void *stream);

/* Masked row softmax followed by dropout (nvFuser issue "HuggingFace
 * BertForMaskedLM - Log Softmax Fusion...", fusion 1, whose outputs include
 * both the probabilities and the dropped, rescaled probabilities):
 *   P[i,t]  as band_softmax (before dropout; P may be NULL if not needed);
 *   Pd[i,t] = f(i,t) * P[i,t], f = 256/(256-t) or 0 the keep-and-scale factor
 *             of the slot's key under the descriptor's dropout (f = 1 when
 *             dropout_p rounds to 0); 0 on unused slots;
 *   lse[i]  as band_softmax (before dropout; may be NULL).
 * The forward product is then O = band_pv(Pd, V); for the backward,
 * band_softmax_bwd with the same descriptor takes P and the gradient of Pd.
 * The keep decisions are recomputed from the descriptor, never stored.
 * No global tokens (SWAB_ERR_UNSUPPORTED); D <= 65536 (else
 * SWAB_ERR_UNSUPPORTED). */
SWAB_API swab_status band_softmax_dropout(const swab_desc *desc, const void *S, void *P, void *Pd,
                                          float *lse, void *stream);

/* AddBiasTranspose (ONNX Runtime issue "[WIP] Improve LongformerAttention
 * performance", item (2): the bias add and the transpose after the merged
 * projection in one kernel, with the widest vector loads, conclusion (g)):
 *   Y[m, bb, hh, i, c] = X[bb, i, m, hh, c] + bias[m, hh, c]
 * for M matrices side by side in each row of X (M = 3: Q, K, V), i.e.
 * X = rows of [b, n, M, h, head_dim] -> Y = M tensors [b, h, n, head_dim].
 * b, h, n, head_dim and dtype come from desc (head_dim * element size a
 * multiple of 16 bytes); the sum is rounded once to the dtype (correctly
 * rounded).  bias ([M, h, head_dim]) may be NULL: a pure transpose.  X, Y,
 * bias device pointers, 16-byte aligned; Y must not overlap X. */
SWAB_API swab_status add_bias_transpose(const swab_desc *desc, int32_t M, const void *X,
                                        const void *bias, void *Y, void *stream);

/* Global queries with their own projections (ONNX Runtime issue "[WIP]
 * Improve LongformerAttention performance", item (3) and its "compact
 * global_q"): the G = desc->n_global global queries, given compact as
 * Qg [b, h, G, 64] (the global_q projection of the global tokens only), attend
 * to every position through separate global key / value projections
 * Kg, Vg [b, h, n, 64]:
 *   Og[g] = sum_j p_gj Vg[j],  p_gj = softmax_j(scale * Qg[g].Kg[j]),
 *   lseg[g] = log sum_j exp(scale * Qg[g].Kg[j])   ([b, h, G] fp32, may be NULL).
 * Together with the band path this gives attention with separate global
 * projections: run the band calls with global_idx (local rows attend to their
 * band keys outside G plus G, with Q, K, V), then replace O's global rows
 * O[G[g]] by Og[g].  In the backward, give the band calls dO with its global
 * rows set to 0 and global_attention_bwd dOg[g] = dO[G[g]].
 * head_dim 64, contiguous layout, no key bias or dropout.  workspace:
 * global_attention_workspace(desc) bytes of device memory, 16-byte aligned,
 * shared by the forward and the backward (not concurrently). */
SWAB_API size_t global_attention_workspace(const swab_desc *desc);
SWAB_API swab_status global_attention(const swab_desc *desc, float scale, const void *Qg,
                                      const void *Kg, const void *Vg, void *Og, float *lseg,
                                      void *workspace, void *stream);
/* Backward of global_attention: with delta_g = dOg[g].Og[g] and
 * ds_gj = p_gj (dOg[g].Vg[j] - delta_g):
 *   dQg = scale ds Kg,  dKg = scale ds^T Qg,  dVg = p^T dOg.
 * lseg is the forward's (required).  dKg, dVg rows have one writer each;
 * dQg sums per-tile partials in a fixed order (bitwise repeatable). */
SWAB_API swab_status global_attention_bwd(const swab_desc *desc, float scale, const void *Qg,
                                          const void *Kg, const void *Vg, const void *Og,
                                          const void *dOg, const float *lseg, void *dQg,
                                          void *dKg, void *dVg, void *workspace, void *stream);

/* Band x dense product (TVM thread, post 6: transpose_t1 = 0, t1d3 = 2w+1):
 *   O[i,c] = alpha * sum over used slots t of P[i,t] * V[j(i,t), c]
 *            (+ alpha * sum_g Pg->cols[i,g] * V[G[g],c]);
 *   a global query's row is alpha * sum_j Pg->rows[g,j] * V[j,c].
 * Forward: O = P.V (alpha = 1).  Backward: dQ = band_pv(alpha, dS, K). */
SWAB_API swab_status band_pv(const swab_desc *desc, float alpha, const void *P,
                             const swab_glob *Pg, const void *V, void *O, void *stream);

/* Transposed band x dense product (TVM thread, post 6: transpose_t1 = 1):
 *   X[j,c] = alpha * sum over (i,t) with j(i,t) = j, t used, of Bd[i,t]*Y[i,c]
 *            (+ global terms of Bg->cols and Bg->rows).
 * band_qk_bwd_t gives dK = alpha * dS^T.Q; band_pv_bwd_t gives
 * dV = P^T.dO (alpha = 1).  The two names run the same kernel.
 * Deterministic: every output row has one writer, no atomics. */
SWAB_API swab_status band_qk_bwd_t(const swab_desc *desc, float alpha, const void *dS,
                                   const swab_glob *dSg, const void *Q, void *dK, void *stream);
SWAB_API swab_status band_pv_bwd_t(const swab_desc *desc, float alpha, const void *P,
                                   const swab_glob *Pg, const void *dO, void *dV, void *stream);

/* Softmax backward on the band (derivative of band_softmax):
 *   dS[i,t] = P[i,t] * (dP[i,t] - delta_i) on used slots, 0 elsewhere,
 *   delta_i = sum over used slots of P*dP (+ sum_g Pg*dPg);
 * global pieces likewise (dSg->cols, dSg->rows).  With the descriptor's
 * dropout (derivative of band_softmax_dropout's Pd): P is the probabilities
 * before dropout, dP the gradient of Pd, and
 *   dS[i,t] = P[i,t] * (f(i,t) dP[i,t] - delta_i), delta_i = sum P*f*dP
 * (D <= 65536, else SWAB_ERR_UNSUPPORTED). */
SWAB_API swab_status band_softmax_bwd(const swab_desc *desc, const void *P, const swab_glob *Pg,
                                      const void *dP, const swab_glob *dPg, void *dS,
                                      const swab_glob *dSg, void *stream);

/* Fused forward: the same O (and lse, may be NULL) as band_qk(scale) ->
 * band_softmax -> band_pv, with the scores kept on chip (never written to
 * memory).  With global tokens (f16 / bf16, contiguous layout, lse required,
 * n <= 188416): local rows attend to their band keys outside G plus G, global
 * rows to every key, as in the materialised calls; computed as the band part
 * (global keys masked), the global columns merged into the local rows by
 * log-sum-exp, and the global rows' dense attention.  fp32 or the strided
 * layout with global tokens: SWAB_ERR_UNSUPPORTED. */
SWAB_API swab_status band_attention(const swab_desc *desc, float scale, const void *Q,
                                    const void *K, const void *V, void *O, float *lse,
                                    void *stream);

/* Fused backward of band_attention: dQ, dK, dV of
 *   O = softmax_band(scale * Q.K^T) . V
 * recomputing the band probabilities on chip from lse (the forward's
 * log-sum-exp) and never writing a band tensor:
 *   P = exp(scale*Q.K^T - lse), dP = dO.V^T, delta_i = dO_i . O_i,
 *   dS = P*(dP - delta), dQ = scale*dS.K, dK = scale*dS^T.Q, dV = P^T.dO
 * on the used slots (the two backward products of the TVM thread, post 6,
 * with the textbook softmax derivative).
 * `workspace` is caller-owned device memory of band_attention_bwd_workspace()
 * bytes, 16-byte aligned; its contents on entry do not matter.  For fp16 /
 * bf16 it holds the per-row delta and an fp32 dQ accumulator: dK and dV have
 * one writer per row, while each key tile's contribution to dQ is added into
 * the accumulator by TMA reduce-add stores (cp.reduce.async.bulk.tensor, fp32
 * additions in the memory system) in an order that varies between runs, so
 * dQ may differ in its last bits from run to run (within the rounding of one
 * fp32 sum; band_attention_bwd_noalloc is bitwise repeatable).  For fp32 it holds the delta only and every output is
 * repeatable.
 * For fp16 / bf16 the call launches three kernels.  The last two are launched
 * as programmatic dependents: they may start while the one before runs and
 * wait inside for what it wrote.  For the caller the call stays ordered on
 * the stream like any kernel launch.
 * Global tokens (f16 / bf16, contiguous layout, no key bias or dropout,
 * n <= 98304; else SWAB_ERR_UNSUPPORTED): the gradients of the attention with
 * global tokens of band_attention -- local rows over their band keys outside G
 * plus G, global rows over every key.  The call then runs the band (global
 * keys and global queries left out), the global columns (every local row
 * against the G global keys, gathered into the workspace) and the global
 * rows (the global_attention_bwd computation with the shared Q, K, V as the
 * global projections), the dK, dV terms of all three added in fp32 before one
 * rounding; the workspace (band_attention_bwd_workspace) then also holds the
 * gathered rows and keys and the global rows' dK, dV terms. */
SWAB_API swab_status band_attention_bwd(const swab_desc *desc, float scale, const void *Q,
                                        const void *K, const void *V, const void *O,
                                        const void *dO, const float *lse, void *dQ, void *dK,
                                        void *dV, void *workspace, void *stream);

/* Bytes of the keep-bit cache (swab_desc.dropout_mask) for `desc`: b*h*n rows
 * of ceil((w + w_upper + 1) / 32) + 1 words (0 if desc is NULL). */
SWAB_API size_t band_attention_dropout_mask_bytes(const swab_desc *desc);

/* Bytes of workspace band_attention_bwd needs for `desc` (0 if desc is NULL):
 * fp16 / bf16: round_up(b*h*n*4, 256) + b*h*n*64*4, plus with global tokens
 * the sections of the gathered global rows, keys and values and the global
 * rows' dK, dV terms (about 2*b*h*n*64*2 bytes more);
 * fp32: round_up(b*h*n*4, 256). */
SWAB_API size_t band_attention_bwd_workspace(const swab_desc *desc);

/* band_attention_bwd for callers that cannot allocate device memory: the same
 * computation and arguments, minus the workspace.  It needs only the per-row
 * delta as scratch because it computes dQ in a kernel of its own (one writer
 * per row) instead of summing it in an fp32 accumulator, so its results agree
 * with band_attention_bwd within rounding and repeat bitwise.  Some callers have
 * no way to obtain a device buffer of their own -- code running under an
 * allocator or memory pool they do not control, plugins handed only input and
 * output pointers, or contexts where a cudaMalloc would synchronise or is
 * forbidden -- so this variant keeps its per-row scratch in a module-scope
 * device array of SWAB_NOALLOC_MAX_ROWS floats (16 MiB), which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated or
 * freed by the call (no cudaMalloc, cudaFree or allocating library routine).
 *   - b*h*n must not exceed SWAB_NOALLOC_MAX_ROWS; larger problems return
 *     SWAB_ERR_UNSUPPORTED (use band_attention_bwd with a workspace).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture.  A first call made while `stream` is being captured
 *     returns SWAB_ERR_UNSUPPORTED and launches nothing.
 *   - The cached address belongs to the device's context at the first call:
 *     resetting the device (cudaDeviceReset) after that call is not
 *     supported, since later calls would use the old address.
 *   - All calls share the one array, which keeps the last call's contents
 *     (every call overwrites what it reads before reading it).  Calls whose
 *     executions overlap on the GPU -- on different streams, or from different
 *     threads without ordering -- race on it; serialise them.
 * The pages have no counterpart for this entry point: it only changes where
 * the library's own scratch lives. */
SWAB_API swab_status band_attention_bwd_noalloc(const swab_desc *desc, float scale, const void *Q,
                                                const void *K, const void *V, const void *O,
                                                const void *dO, const float *lse, void *dQ,
                                                void *dK, void *dV, void *stream);

/* Human-readable name of a status code (static string). */
SWAB_API const char *swab_status_string(swab_status status);

/* Reads (and, if reset != 0, clears) the library's device status word on the
 * current device: bit k set means SWAB status k was raised by a kernel.
 * Synchronises the device.  Returns SWAB_ERR_CUDA if the read fails. */
SWAB_API swab_status swab_device_status(int32_t *flags, int32_t reset);

/* Failure-detection self-test: launches one warp that waits on an mbarrier no
 * thread ever arrives at, using the same bounded wait as every pipelined
 * kernel, with a limit of `limit_us` microseconds (1..1000000).  The wait gives
 * up, records SWAB_ERR_TIMEOUT in the device status word and the kernel
 * returns; nothing faults or hangs and the context stays usable.  Read the
 * result with swab_device_status().  No counterpart on the pages: it tests
 * the library's own error reporting. */
SWAB_API swab_status swab_selftest_wait_timeout(uint32_t limit_us, void *stream);

/* ---------------------------------------------------------------------------
 * Bounds-checked build.  The library also builds as libswab_bounds.so with
 * SWAB_BOUNDS_CHECK=1: the same kernels, in which every plain global load,
 * store and reduction first tests the bytes it touches against the extents of
 * the call's buffers.  The host derives those extents from the descriptor and
 * the documented shapes (dense [b, h, n, hd] or rows of [b, n, row_stride];
 * band [b*h, n, D]; companions, lse, key bias, keep-bit cache and workspace by
 * their sizes above), plus the library's own device arrays.  An access outside
 * all of them is not made (a store is dropped, a load reads a scratch line):
 * the kernel raises SWAB_ERR_BOUNDS in the device status word, records the
 * first such access (swab_bounds_report) and runs on.  TMA copies are clipped
 * by the hardware to their tensor map; the host checks each map's footprint
 * against the same extents before launching and returns SWAB_ERR_BOUNDS (no
 * launch) if one overhangs.  No counterpart on the pages: it stands in for a
 * memory checker where none can run.  The checked build is slower; its
 * results are the regular build's, bit for bit.
 * ------------------------------------------------------------------------- */

/* 1 in the bounds-checked build, 0 in the regular one. */
SWAB_API int32_t swab_bounds_checked(void);

/* First out-of-bounds access recorded on the current device since the last
 * reset: out[0] = source site (file id << 16 | line) + 1, 0 if none;
 * out[1] = its address; out[2] = its size in bytes.  Synchronises the device;
 * reset != 0 clears the record.  Always zero in the regular build. */
SWAB_API swab_status swab_bounds_report(uint64_t *out, int32_t reset);

/* Self-test of the bounds checks (checked build only, SWAB_ERR_UNSUPPORTED
 * otherwise): one warp stores through the check into a library-owned device
 * array of 128 floats with an extent table that covers only its first 64.
 * Lane l stores to element l (inside the extent) and to element 64 + l
 * (valid memory outside it).  Synchronises `stream`; returns SWAB_OK when the
 * stores inside landed and the ones outside did not (else SWAB_ERR_BOUNDS).
 * The refused stores also raise SWAB_ERR_BOUNDS in the device status word and
 * are recorded (swab_bounds_report).  Nothing outside the array is ever
 * addressed. */
SWAB_API swab_status swab_selftest_bounds(void *stream);

/* Library version, e.g. "0.1.0". */
SWAB_API const char *swab_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWAB_H */
