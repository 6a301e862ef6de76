/*
 * moe.h -- C ABI of libmoe_gb300: one top-k Mixture-of-Experts FFN layer with
 * SwiGLU experts, forward and backward, on one GB300 (sm_103a).  Dropless by
 * default; optionally with a per-expert capacity (token dropping) and, for the
 * dispatch step alone, a local expert range (the "scatter & drop" that follows
 * an all-gather of every token).
 *
 * The layer (sources named by page title and section):
 *   - a trainable gate scores every expert per token; the k experts with the
 *     highest probability are chosen and their outputs summed, weighted
 *     (DisagMoE, §2.1 "混合专家（MoE）结构");
 *   - token copies are sorted by expert, then by source, so that each expert's
 *     rows are contiguous (MegaScale-MoE research digest, §3.3 under Diagram C);
 *   - the experts are SwiGLU FFNs run together as one GroupedGEMM, "one kernel
 *     for the matrix products of several experts" (digest, glossary; MegaScale-
 *     MoE paper review, §三 核心公式 and 训练流程);
 *   - forward and backward are explicit operators, not autograd (digest §3.3);
 *   - load balance may drop tokens per GPU (digest §3.2, the paragraph after
 *     Figure 7), and the all-gather path of adaptive EP drops, locally, the
 *     tokens that no local expert takes (digest §3.2, Diagram B; review §四
 *     自适应EP通信策略详解, step 2).
 *
 * Conventions shared by every entry point
 *   - Pointers named x, Wg, W1 ... and every output are DEVICE pointers owned by
 *     the caller.  The library never allocates device memory and never frees
 *     any.  Scratch space is the caller's `ws` buffer of at least
 *     moe_workspace_bytes() bytes; the layer context is the caller's `saved`
 *     buffer of moe_saved_bytes() bytes.  Every pointer must be 16-byte
 *     aligned; ws and saved must be 256-byte aligned.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream); the
 *     library never synchronises except in moe_read_device_status().
 *   - All matrices are row-major and dense:
 *       x, dy, y, dx : [T, h]   bf16        Wg, dWg : [h, E] fp32    b : [E] fp32
 *       W1, W3       : [E, h, f] bf16       W2      : [E, f, h] bf16
 *       dW1, dW3     : [E, h, f] fp32       dW2     : [E, f, h] fp32
 *       topk_idx     : [T, k] int32         gates   : [T, k] fp32
 *     An assignment a = t*k + j is token t's j-th chosen expert.  A permuted
 *     row p indexes the expert-major order: rows offsets[e] .. offsets[e+1]-1
 *     belong to expert e, in ascending a.
 *   - Token dropping (dims.capacity = C > 0): expert e takes only its first C
 *     assignments in ascending a; every other assignment is dropped.  A
 *     dropped assignment has perm_dst[a] = -1, adds nothing to y and gets no
 *     gradient through the experts (its gate gradient is 0); the gates are
 *     not renormalised.  Only the offsets[E] <= T*k placed rows exist: rows
 *     p >= offsets[E] of the permuted buffers are neither written nor read.
 *     C = 0 is dropless (offsets[E] = T*k).
 *   - Gradients are written, not accumulated.  An expert that receives no
 *     token gets zero weight gradients.
 *   - Argument errors are found on the host before any launch and returned as
 *     a status; nothing is launched then.  CUDA launch errors return
 *     MOE_ERR_CUDA.  Device code never traps or prints: a kernel whose bounded
 *     wait runs out records MOE_ERR_DEVICE_TIMEOUT in the status word at the
 *     start of `ws` and returns; moe_read_device_status() reports it.  A
 *     kernel that reads an index from device memory (an expert id in
 *     topk_idx, an entry of perm_src or perm_dst, an expert offset handed in
 *     by the caller) checks it: one out of range is recorded as
 *     MOE_ERR_DEVICE_INDEX in the same status word and that element is
 *     skipped (an assignment not placed, a zero row, a slot that adds
 *     nothing), so nothing is read or written out of bounds.  The calls that
 *     take no workspace (moe_combine, moe_unpermute, moe_quantize_rows_fp8,
 *     moe_permute_noalloc) record into one status word per device that the
 *     library keeps (its address is looked up on the first such call on a
 *     device and kept until the process exits); moe_read_device_status(NULL,
 *     stream) reports that one.
 *   - Supported shapes: 1 <= k <= 8, E <= 64, T*k < 2^31, h and f multiples
 *     of 64 (the GEMMs' K blocks are 64 wide).  Calls that choose experts
 *     (moe_route, moe_layer_fwd/bwd, moe_saved_bytes) also need k <= E; the
 *     others may run on a subset of the experts (E = a local expert count).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t;   /* == cudaStream_t */
typedef struct CUevent_st* moe_event_t;     /* == cudaEvent_t */
typedef uint16_t moe_bf16;                  /* bf16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad dimension */
  MOE_ERR_UNSUPPORTED = 2,     /* shape outside the supported set */
  MOE_ERR_WORKSPACE = 3,       /* ws_bytes smaller than required */
  MOE_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_TIMEOUT = 5,  /* a kernel's bounded wait ran out */
  MOE_ERR_DEVICE_INDEX = 6     /* an index read on the device was out of range */
} moe_status;

typedef struct {
  int32_t T;         /* tokens */
  int32_t h;         /* hidden size */
  int32_t f;         /* expert FFN width (h_ffn) */
  int32_t E;         /* experts */
  int32_t k;         /* experts per token */
  int32_t has_bias;  /* 1: router bias b[E] is added to the logits */
  int32_t capacity;  /* 0: dropless; C > 0: at most C assignments per expert */
  int32_t sar;       /* 1: selective activation rematerialisation (see below) */
} moe_dims;

typedef enum {
  MOE_OP_ROUTE = 0,
  MOE_OP_PERMUTE = 1,
  MOE_OP_EXPERT_FFN_FWD = 2,
  MOE_OP_EXPERT_FFN_BWD = 3,
  MOE_OP_ROUTER_BWD = 4,
  MOE_OP_LAYER_FWD = 5,
  MOE_OP_LAYER_BWD = 6,
  MOE_OP_LAYER_FWD_FP8 = 7,
  MOE_OP_LAYER_BWD_FP8 = 8
} moe_op;

/* Per-expert capacity for a capacity factor: ceil(factor * T * k / E), the
 * share of the T*k assignments an expert gets under perfect balance times the
 * factor (the digest's per-GPU token dropping for load balance, §3.2 after
 * Figure 7; the factor is the usual way to size it).  Returns the value for
 * dims.capacity, or -1 when T < 0, k < 1, E < 1, factor <= 0 or the result
 * does not fit an int32. */
int32_t moe_capacity_for(int32_t T, int32_t k, int32_t E, double factor);

/* Scratch bytes entry point `op` needs for `dims` (0 on invalid dims).  The
 * first 256 bytes of every workspace hold the device status word; zero the
 * workspace once before first use (or call moe_clear_device_status). */
size_t moe_workspace_bytes(const moe_dims* dims, int op);

/* Bytes of the forward->backward context that moe_layer_fwd writes into
 * `saved` and moe_layer_bwd reads: routing, dispatch maps and activations.
 *   sar = 0: the permuted token rows x_perm and all four expert activations
 *            A = X W1, B = X W3, H = silu(A)*B, O = H W2; per layer
 *            (2k + 3k f/h) T h bf16 elements.
 *   sar = 1: selective activation rematerialisation (digest §3.3 "Inter-
 *            operator overlap"; review 选择性激活重计算): only A and B, i.e.
 *            2k (f/h) T h elements -- the pages' (2kf + ...) bsh/n after SAR,
 *            against (... 2k + 3kf ...) bsh/n before, at n = 1.  The backward
 *            gathers x_perm and dy again, rebuilds H from A and B inside the
 *            FC2 dgrad, and takes the gate gradient <dy, O> as <H, dy W2^T>
 *            (the same value), so O is never needed.  H, O and x_perm then live
 *            in the forward workspace, which is not kept between the calls. */
size_t moe_saved_bytes(const moe_dims* dims);

/* Router logits l = x Wg (+ b), softmax over the E experts, top-k selection
 * (descending logit, ties to the lower expert id) and renormalisation of the
 * k probabilities: gates[t,j] = p[e_j] / sum_j' p[e_j'].  DisagMoE §2.1.
 * In: x [T,h] bf16, Wg [h,E] fp32, b [E] fp32 (ignored unless has_bias).
 * Out: topk_idx [T,k] int32, gates [T,k] fp32.  Logits accumulate in fp32. */
moe_status moe_route(const moe_dims* dims, const moe_bf16* x, const float* Wg,
                     const float* b, int32_t* topk_idx, float* gates,
                     void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch: per-expert histogram, exclusive scan and the stable expert-major
 * permutation (digest §3.3: sorted by expert, then by source; review §四:
 * the scatter that makes each expert's tokens contiguous).  Deterministic,
 * no atomics.
 * In: topk_idx [T,k]; x [T,h] bf16 or NULL.
 * Out: counts [E], offsets [E+1] (offsets[E] = T*k when dropless), perm_src
 * [T*k] (permuted row -> assignment; the first offsets[E] entries are
 * written), perm_dst [T*k] (assignment -> permuted row, -1 if dropped), and,
 * when x and x_perm are both non-NULL, x_perm [T*k,h] with
 * x_perm[p] = x[perm_src[p] / k] for p < offsets[E]. */
moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx,
                       const moe_bf16* x, int32_t* counts, int32_t* offsets,
                       int32_t* perm_src, int32_t* perm_dst, moe_bf16* x_perm,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_permute with no workspace argument (the pages have no counterpart; this
 * is an interface convenience).  For callers that cannot allocate device
 * memory when they dispatch, such as a runtime that owns a fixed memory
 * budget.  Same arguments
 * and outputs as moe_permute minus ws/ws_bytes.  Its scratch is a 1 MiB array
 * in the library's device memory (held by every GPU that loads the library
 * until exit), so it supports ceil(T*k / 1024) * E <= 131072 and returns
 * MOE_ERR_UNSUPPORTED beyond that.  The first call on a device looks up the
 * array's device address (a host-side runtime query).  The address is kept
 * for the life of the process: after a cudaDeviceReset, restart the
 * process before calling this again.  All calls share the array: calls that
 * overlap on the GPU race.  Index errors (an expert id out of range) go to the
 * per-device status word of the calls without a workspace.  Allocates
 * nothing. */
moe_status moe_permute_noalloc(const moe_dims* dims, const int32_t* topk_idx,
                               const moe_bf16* x, int32_t* counts,
                               int32_t* offsets, int32_t* perm_src,
                               int32_t* perm_dst, moe_bf16* x_perm,
                               moe_stream_t stream);

/* The all-gather path's local "scatter & drop" (digest §3.2, Diagram B; review
 * §四 自适应EP通信策略详解, step 2): given every token's routing, place only the
 * assignments to the local experts e_lo <= e < e_hi (0 <= e_lo < e_hi <= E),
 * each expert taking at most dims.capacity of them when that is non-zero.
 * Same outputs as moe_permute over the EL = e_hi - e_lo local experts:
 * counts [EL], offsets [EL+1] (local expert i = global e_lo + i), perm_src
 * [T*k] (first offsets[EL] entries), perm_dst [T*k] (-1 for every assignment
 * not placed here), x_perm rows p < offsets[EL] when x and x_perm are given.
 * The local rows then run through moe_expert_ffn_fwd/bwd with dims.E = EL and
 * the local experts' weights; moe_combine with this perm_dst gives the local
 * experts' share of y (the partial sum the reduce-scatter adds up).
 * Workspace: moe_workspace_bytes(dims, MOE_OP_PERMUTE). */
moe_status moe_permute_local(const moe_dims* dims, const int32_t* topk_idx,
                             int32_t e_lo, int32_t e_hi, const moe_bf16* x,
                             int32_t* counts, int32_t* offsets,
                             int32_t* perm_src, int32_t* perm_dst,
                             moe_bf16* x_perm, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Inverse row move: rows_assign[a] = rows_perm[perm_dst[a]] for a < T*k, a
 * zero row where perm_dst[a] = -1.  rows_perm, rows_assign: [T*k, h] bf16.
 * It undoes the expert-major order of the dispatch (digest §3.3: token copies
 * sorted by expert, then by source), taking rows back to assignment order
 * a = t*k + j.  A perm_dst entry >= T*k gives a zero row and is recorded as
 * MOE_ERR_DEVICE_INDEX in the per-device status word (no workspace; see
 * moe_read_device_status). */
moe_status moe_unpermute(const moe_dims* dims, const int32_t* perm_dst,
                         const moe_bf16* rows_perm, moe_bf16* rows_assign,
                         moe_stream_t stream);

/* Expert SwiGLU FFN as GroupedGEMMs over the expert-contiguous rows:
 * for each e and rows p of e, with X[p] = x[perm_src[p] / k]:
 *   A = X W1[e],  B = X W3[e],  H = silu(A) * B,  O = H W2[e]
 * (review §三 核心公式: SwiGLU with MoE, 3k*bsh*h_ffn multiply-adds).
 * bf16 operands, fp32 accumulation in tensor memory; A, B, H, O stored bf16
 * [T*k, f] / [T*k, h], rows p < offsets[E] only.  offsets is read on the
 * device only. */
moe_status moe_expert_ffn_fwd(const moe_dims* dims, const moe_bf16* x,
                              const int32_t* perm_src, const int32_t* offsets,
                              const moe_bf16* W1, const moe_bf16* W3,
                              const moe_bf16* W2, moe_bf16* A, moe_bf16* B,
                              moe_bf16* H, moe_bf16* O,
                              void* ws, size_t ws_bytes, moe_stream_t stream);

/* Gate-weighted combine: y[t] = sum_{j<k} gates[t,j] * O[perm_dst[t*k+j]],
 * summed in fp32 in slot order, rounded once to bf16; slots with
 * perm_dst = -1 are skipped.  Deterministic (a gather, no scatter-add).
 * DisagMoE §2.1 (weighted sum). */
moe_status moe_combine(const moe_dims* dims, const moe_bf16* O,
                       const float* gates, const int32_t* perm_dst,
                       moe_bf16* y, moe_stream_t stream);

/* Backward of the expert FFN for the loss gradient dy [T,h]:
 *   dO[p] = gates[a] * dy[t]          (a = perm_src[p], t = a / k)
 *   dg[a] = <dy[t], O[p]>             (gradient of the gate, fp32 [T*k])
 *   dH = dO W2[e]^T ; dA = dH * B * s (1 + A (1 - s)), s = sigmoid(A) ;
 *   dB = dH * silu(A)
 *   dW2[e] = H_e^T dO_e ; dW1[e] = X_e^T dA_e ; dW3[e] = X_e^T dB_e
 *   dX_perm = dA W1[e]^T + dB W3[e]^T          (fp32 [T*k, h])
 * FC2's gradients take fc2_in = H and the gradient of fc2_out (review
 * 选择性激活重计算).  A, B, H, O are moe_expert_ffn_fwd's outputs.  Rows
 * p < offsets[E] only: dg[a] is written for the placed assignments
 * a = perm_src[p] alone, and so are the dX_perm rows. */
moe_status moe_expert_ffn_bwd(const moe_dims* dims, const moe_bf16* x,
                              const moe_bf16* dy, const float* gates,
                              const int32_t* perm_src, const int32_t* offsets,
                              const moe_bf16* W1, const moe_bf16* W3,
                              const moe_bf16* W2, const moe_bf16* A,
                              const moe_bf16* B, const moe_bf16* H,
                              const moe_bf16* O, float* dX_perm, float* dg,
                              float* dW1, float* dW3, float* dW2,
                              void* ws, size_t ws_bytes, moe_stream_t stream);

/* Router backward and the token gradient:
 *   dl[t,j] = g_j (dg_j - sum_i g_i dg_i)     (softmax over the k selected),
 *             evaluated as g_j sum_i g_i (dg_j - dg_i) since sum_i g_i = 1
 *   dx[t]   = sum_j dX_perm[perm_dst[t*k+j]] + sum_j dl[t,j] Wg[:, e_j]  (bf16)
 *   dWg     = x^T dl (fp32 [h,E]; a fixed-order two-level reduction)
 * In: x, Wg, topk_idx, gates, dg [T*k], dX_perm [T*k,h] fp32, perm_src,
 * perm_dst, offsets.  A slot with perm_dst = -1 counts with dg = 0 and adds
 * no dX_perm row. */
moe_status moe_router_bwd(const moe_dims* dims, const moe_bf16* x,
                          const float* Wg, const int32_t* topk_idx,
                          const float* gates, const float* dg,
                          const float* dX_perm, const int32_t* perm_src,
                          const int32_t* perm_dst, const int32_t* offsets,
                          moe_bf16* dx, float* dWg,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* Whole layer forward: route, permute, expert FFN, combine.  Writes y [T,h]
 * and the context `saved` (moe_saved_bytes) for moe_layer_bwd. */
moe_status moe_layer_fwd(const moe_dims* dims, const moe_bf16* x,
                         const float* Wg, const float* b, const moe_bf16* W1,
                         const moe_bf16* W3, const moe_bf16* W2, moe_bf16* y,
                         void* saved, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* ---------------------------------------------------------------- FP8
 * FP8 training with per-token quantisation instead of per-tensor (review §三
 * 创新点 "FP8训练优化"; digest §3.4).  The expert forward matmuls run on e4m3
 * codes (tcgen05 kind::f8f6f4) with float32 scales:
 *   activations x_perm and H: one scale per row, s = amax(|row|) / 448;
 *   weights: one scale per output column of each expert (amax over the
 *   contraction dimension);
 * q = e4m3(v / s) with an IEEE float32 division and round-to-nearest-even,
 * saturating at 448; s = 1 for an all-zero row or column.  The matmul sums
 * the exact code products in fp32 and multiplies by s_row * s_col.  H is
 * quantised from its bf16 copy.  The backward is the bf16 moe_layer_bwd on
 * the activations (A, B, H, O) this forward stores.  Requires h and f to be
 * multiples of 128 (MOE_ERR_UNSUPPORTED otherwise). */

/* Bytes of a quantised-weight buffer `qw` (0 on invalid or unsupported dims). */
size_t moe_fp8_weight_bytes(const moe_dims* dims);

/* Quantises the expert weights into `qw` (256-byte aligned, caller-owned):
 *   "W13q" [E, 2f, h] e4m3, K-major: per expert, 128-row groups alternating
 *          W1 columns and W3 columns (group 2j: W1[:, 128j + r], group 2j+1:
 *          W3[:, 128j + r], r < 128; each row holds the h codes of a column);
 *   "W2q"  [E, h, f] e4m3, K-major (row n holds the f codes of W2[:, n]);
 *   "s1", "s3" [E, f] and "s2" [E, h] float32 column scales.
 * Call it after every update of W1, W3, W2; moe_fp8_weight_view(name) gives
 * each part's device address. */
moe_status moe_quantize_weights_fp8(const moe_dims* dims, const moe_bf16* W1,
                                    const moe_bf16* W3, const moe_bf16* W2,
                                    void* qw, moe_stream_t stream);
void* moe_fp8_weight_view(const moe_dims* dims, void* qw, const char* name);

/* Row quantisation on its own: for p < rows, with src = idx[p] / div (or p
 * when idx is NULL; then src_rows >= rows), q[p, :] = e4m3(in[src, :] / s[p]),
 * s[p] = amax(|in[src, :]|) / 448.  in [src_rows, n] bf16, q [rows, n] bytes,
 * scale [rows] float32; n a multiple of 16. */
moe_status moe_quantize_rows_fp8(const moe_bf16* in, int64_t rows, int32_t n,
                                 const int32_t* idx, int32_t div,
                                 int64_t src_rows, uint8_t* q, float* scale,
                                 moe_stream_t stream);

/* moe_layer_fwd with the FP8 expert forward: route, dispatch, per-token
 * quantisation of the permuted rows, FC1 (+SwiGLU) on e4m3 codes, per-token
 * quantisation of H, FC2 on e4m3 codes, combine.  Weights come only from
 * `qw` (moe_quantize_weights_fp8).  Writes y and the same `saved` context as
 * moe_layer_fwd (A, B, H, O from the FP8 matmuls), for moe_layer_bwd.
 * dims.sar = 1 is MOE_ERR_UNSUPPORTED here: the sar backward takes the gate
 * gradient <dy, O> as <H, dy W2^T>, which needs O = H W2 exactly, and this
 * O comes from the e4m3 codes of H and W2.
 * Workspace: moe_workspace_bytes(dims, MOE_OP_LAYER_FWD_FP8). */
moe_status moe_layer_fwd_fp8(const moe_dims* dims, const moe_bf16* x,
                             const float* Wg, const float* b, const void* qw,
                             moe_bf16* y, void* saved, void* ws,
                             size_t ws_bytes, moe_stream_t stream);

/* FP8 data gradient of the backward, with the same per-token reading: the
 * FC1 dgrad dX = dA W1^T + dB W3^T runs on e4m3 codes as one contraction
 * over both halves, so a row of dA and the same row of dB share one scale
 * (their amax is recorded by the FC2 dgrad's epilogue) and row n of W1[e] and
 * row n of W3[e] share one.  FC2 dgrad stays bf16: its cost is the fused
 * SwiGLU backward in its epilogue, which e4m3 operands do not shorten
 * (measured).  The weight gradients stay bf16 matmuls on the bf16 dO, dA,
 * dB.  Requires h, f multiples of 128 and dims.sar = 0.
 *
 * moe_quantize_weights_fp8_bwd writes into `qwb` (256-byte aligned,
 * moe_fp8_bwd_weight_bytes): "W1r", "W3r" [E, h, f] e4m3 (row n of W1[e] and
 * of W3[e] with one shared scale) and "s13r" [E, h] float32;
 * moe_fp8_bwd_weight_view gives each part's address.  Call it after every
 * weight update. */
size_t moe_fp8_bwd_weight_bytes(const moe_dims* dims);
moe_status moe_quantize_weights_fp8_bwd(const moe_dims* dims,
                                        const moe_bf16* W1, const moe_bf16* W3,
                                        void* qwb, moe_stream_t stream);
void* moe_fp8_bwd_weight_view(const moe_dims* dims, void* qwb,
                              const char* name);

/* moe_layer_bwd with the FP8 FC1 data gradient above, from a `saved` context
 * of moe_layer_fwd or moe_layer_fwd_fp8 (sar = 0).  W2 (bf16) feeds the FC2
 * dgrad.  Same outputs as moe_layer_bwd.  Workspace:
 * moe_workspace_bytes(dims, MOE_OP_LAYER_BWD_FP8). */
moe_status moe_layer_bwd_fp8(const moe_dims* dims, const moe_bf16* x,
                             const moe_bf16* dy, const float* Wg,
                             const moe_bf16* W2, const void* qwb,
                             const void* saved, moe_bf16* dx, float* dWg,
                             float* dW1, float* dW3, float* dW2, void* ws,
                             size_t ws_bytes, moe_stream_t stream);

/* Whole layer backward from `saved`: writes dx [T,h] bf16 and the fp32
 * gradients dWg, dW1, dW3, dW2.  The router bias gets no gradient. */
moe_status moe_layer_bwd(const moe_dims* dims, const moe_bf16* x,
                         const moe_bf16* dy, const float* Wg,
                         const moe_bf16* W1, const moe_bf16* W3,
                         const moe_bf16* W2, const void* saved, moe_bf16* dx,
                         float* dWg, float* dW1, float* dW3, float* dW2,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* Views into a `saved` context (device pointers at fixed offsets; NULL on
 * invalid dims, and for "x_perm", "H", "O" when dims.sar = 1).  Names:
 * "topk_idx", "gates", "counts", "offsets", "perm_src", "perm_dst",
 * "x_perm", "A", "B", "H", "O". */
void* moe_saved_view(const moe_dims* dims, void* saved, const char* name);

/* Human-readable name of a status. */
const char* moe_status_string(moe_status status);

/* Synchronises `stream`, returns the status word at the start of `ws` and
 * clears it.  ws = NULL: the status word of the calls that take no workspace
 * (moe_combine, moe_unpermute, moe_quantize_rows_fp8, moe_permute_noalloc) on
 * the current device.
 * MOE_ERR_CUDA if the synchronisation itself failed. */
moe_status moe_read_device_status(void* ws, moe_stream_t stream);

/* Zeroes the status word at the start of `ws` (asynchronous); ws = NULL: the
 * current device's status word of the calls without a workspace. */
moe_status moe_clear_device_status(void* ws, moe_stream_t stream);

/* Failure-path self test: launches one thread that waits on an mbarrier
 * nothing will complete, with the same bounded wait the matmul pipelines use
 * but a limit of limit_us microseconds (1 .. 1000000).  The wait gives up,
 * records MOE_ERR_DEVICE_TIMEOUT in the status word at the start of `ws` and
 * the kernel returns; the context stays usable.  No fault, trap or hang. */
moe_status moe_selftest_wait_timeout(void* ws, uint32_t limit_us, moe_stream_t stream);

/* Measurement hook: while `events` is non-NULL, every kernel the library
 * launches from this host thread is followed by cudaEventRecord of the next
 * event on the launching stream (up to `capacity`).  Pass NULL to stop; the
 * return value is the number of events recorded since the previous call.
 * moe_profile_kernel_name(i) names the kernel recorded by event i. */
int moe_profile_events(moe_event_t* events, int capacity);
const char* moe_profile_kernel_name(int i);

/* Number of CUDA kernels the library has launched from the calling host
 * thread since it was loaded (a named step of the measurement hook may launch
 * more than one kernel: the router and the router weight gradient run two). */
int64_t moe_kernel_launches(void);

/* Failure-injection hook for tests: the n-th kernel launch from now on the
 * calling host thread is reported as failed (cudaErrorLaunchFailure), so the
 * entry point that made it returns MOE_ERR_CUDA at that point without
 * launching the rest of its sequence.  The kernel itself runs normally and no
 * device state is touched: the failure exists only on the host.  n <= 0
 * clears a pending injection; the hook clears itself once it fires. */
void moe_test_fail_launch_after(int n);

/* Library build string (arch, version). */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
