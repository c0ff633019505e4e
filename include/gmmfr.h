/*
 * gmmfr — MXFP8 grouped matmul + finalize routing on one GB300 (sm_103a).
 *
 * The operator (grouped_matmul_finalize_routing MXFP8 write-up, czykbl.com/news/94077,
 * sections 2.1-2.2 and 3.1; aclnnGroupedMatmulFinalizeRoutingV3, "计算公式" items 1-4):
 *
 *   for each expert e, for each routed token t in e's range and each column n:
 *     mm(t,n)  = sum_k fp8(x1[t,k]) 2^(pertoken_scale[t,k/64,(k/32)%2]-127)
 *                     * fp8(x2[e,k,n]) 2^(scale[k/64,n,(k/32)%2]-127)        (stage 1)
 *     out[row_index[t], n] += logit[t] * mm(t,n)                             (stages 2, 3)
 *   out[shared_input_offset + i, n] += shared_input_weight * shared_input[i, n]  (stage 4)
 *
 * One E8M0 scale covers 32 consecutive K elements; the [ceil(K/64), 2] pair
 * layout is read as pair k/64, half (k/32)%2 (the write-up's golden expands
 * scales by 32 along K, section 6.3).
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE memory owned by the caller, dense and row-major:
 *     views (gmmfr_tensor, checked against the problem) for the operator and the
 *     weight preparation, plain pointers for the routing step and the FFN, whose
 *     problem structs give every size; the library keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued on it; no entry point synchronises unless it says so.
 *   - A call that returns an error status enqueues no work.  The message of the
 *     last error on the calling thread is available from gmmfr_last_error().
 *   - No entry point allocates device memory: scratch space is the caller's
 *     `workspace`, and prepared weights live in a caller buffer.
 */
#ifndef GMMFR_H
#define GMMFR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GMMFR_API __attribute__((visibility("default")))
#else
#define GMMFR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GMMFR_OK = 0,
  GMMFR_ERR_INVALID_ARG = 1, /* a size, pointer, dtype code or offset is out of range */
  GMMFR_ERR_UNSUPPORTED = 2, /* valid for the operator but not handled here (e.g. a first static-scratch call inside a capture) */
  GMMFR_ERR_WORKSPACE = 3,   /* workspace or prepared buffer too small or misaligned */
  GMMFR_ERR_CUDA = 4,        /* a CUDA runtime call failed (no device, launch error, ...) */
  GMMFR_ERR_DEVICE = 5       /* a device-side check failed; see gmmfr_check_device_errors */
} gmmfr_status;

/* Element formats of x1 and x2: FP8 E4M3/E5M2 (section 3.1), or FP4 E2M1 for the
 * MXFP4 scenario (aclnn V3, Atlas 350) stored two codes per byte along the row's
 * contiguous dimension (K for x1 and a transposed x2, N for a non-transposed x2),
 * the even element in the low nibble; K, and N for a non-transposed E2M1 x2, even
 * (aclnn: "k must be even; n even when x2 is not transposed").  When x1 and x2 are
 * both E2M1 and K % 32 == 0 they stay packed and run on the FP4 block-scaled MMA
 * (kind::mxf4, 256 K elements per tile).  Otherwise an E2M1 operand is expanded exactly
 * to E4M3 (weights at preparation, tokens per call) and runs on the FP8 block-scaled MMA
 * beside the other operand's FP8 codes. */
typedef enum { GMMFR_E4M3 = 0, GMMFR_E5M2 = 1, GMMFR_E2M1 = 2 } gmmfr_fp8_format;

/* Integer type of row_index: int64 as in the tensor table, or int32. */
typedef enum { GMMFR_INDEX_I64 = 0, GMMFR_INDEX_I32 = 1 } gmmfr_index_type;

/* problem.flags */
#define GMMFR_DETERMINISTIC 1u /* row-ordered combine; bit-identical results run to run */

/* Bits of the device error word (gmmfr_check_device_errors). */
#define GMMFR_DEV_BAD_GROUP_LIST 1u /* negative count, decreasing prefix sum, or total > M; ranges were clamped */
#define GMMFR_DEV_BAD_ROW_INDEX 2u  /* a routed token had row_index outside [0, batch); it was skipped */
#define GMMFR_DEV_TIMEOUT 4u        /* a pipeline wait gave up; the output is incomplete */
#define GMMFR_DEV_BAD_EXPERT_ID 8u  /* routing: a top-k expert id outside [0, E); that entry was routed nowhere */

/*
 * Tensor views.  Every tensor argument of the operator is passed as a non-owning view of
 * dense device memory, so that the library can refuse a tensor whose rank, shape, element
 * type or layout does not match the problem (as the aclnn operator checks its aclTensor
 * arguments, "参数说明" / "约束说明") before anything is enqueued, instead of reading past
 * its end.
 *   data     device address; NULL only for a tensor with no elements
 *   dtype    gmmfr_dtype.  FP8, E2M1 and E8M0 tensors may also be passed as raw bytes
 *            (GMMFR_DT_U8); the problem's formats say how the bytes are read
 *   ndim     1 .. 4
 *   shape    in elements of dtype; packed E2M1 (GMMFR_DT_E2M1X2, or U8 holding E2M1 codes)
 *            counts bytes, i.e. pairs of codes, along its packed dimension
 *   strides  in elements; only dense row-major layouts are accepted (the last stride 1,
 *            each other stride the product of the sizes after it; a dimension of size 1
 *            may have any stride)
 * A NULL view pointer means the tensor is absent (an optional input, or x2 and scale when
 * prepared weights are given).
 */
typedef enum {
  GMMFR_DT_U8 = 0,     /* raw bytes */
  GMMFR_DT_E4M3 = 1,   /* FP8 E4M3FN */
  GMMFR_DT_E5M2 = 2,   /* FP8 E5M2 */
  GMMFR_DT_E2M1X2 = 3, /* two FP4 E2M1 codes per byte, the even element in the low nibble */
  GMMFR_DT_E8M0 = 4,   /* E8M0 scale bytes, 2^(b-127) */
  GMMFR_DT_I64 = 5,
  GMMFR_DT_I32 = 6,
  GMMFR_DT_F32 = 7,
  GMMFR_DT_BF16 = 8
} gmmfr_dtype;

#define GMMFR_MAX_DIMS 4
typedef struct {
  void* data;
  int32_t dtype;
  int32_t ndim;
  int64_t shape[GMMFR_MAX_DIMS];
  int64_t strides[GMMFR_MAX_DIMS];
} gmmfr_tensor;

/*
 * Sizes, formats and scalar arguments of one call (section 3.1 tensor table and
 * section 5.1 FinalizeRoutingConfig fields).
 *
 *   M      rows of x1, pertoken_scale, logit, row_index (routed tokens, batch*topk); M >= 0
 *   K      contraction length, K >= 1; even when E2M1 codes are packed along K (an E2M1 x1,
 *          or a transposed E2M1 x2)
 *   N      output columns, N >= 0
 *   E      experts, 1 <= E <= 1024 (aclnn V3 constraint "e <= 1024")
 *   batch  rows of out, batch >= 0
 *   x1_format, x2_format     gmmfr_fp8_format of x1 and x2
 *   transpose_x2             0: x2 [E,K,N], scale [ceil(K/64),N,2];
 *                            1: x2 [E,N,K], scale [N,ceil(K/64),2] (scale follows x2, section 5.3)
 *   scale_per_expert         1: scale carries a leading [E] dimension (aclnn's 4-D form)
 *   group_list_type          0: prefix sums, expert e owns [g[e-1], g[e]) with g[-1] = 0;
 *                            1: counts, expert e owns [sum g[:e], sum g[:e] + g[e]) (section 4.3)
 *   row_index_type           gmmfr_index_type
 *   shared_rows              rows of shared_input (0: no shared input)
 *   shared_offset            first out row of the shared add; 0 <= offset, offset + rows <= batch
 *   shared_weight            multiplier of shared_input (default 1.0 on the page)
 *   flags                    GMMFR_DETERMINISTIC or 0
 *   expected_tokens_per_expert  tiling hint (aclnn V3 tuningConfigOptional, first value: the
 *                            expected tokens per expert); 0 = none.  When > 0 it fixes the
 *                            token group width (32, 64 or 128, the smallest that holds it)
 *                            instead of deriving it from the largest expert on the device.
 */
typedef struct {
  int64_t M, K, N, E, batch;
  int32_t x1_format, x2_format;
  int32_t transpose_x2;
  int32_t scale_per_expert;
  int32_t group_list_type;
  int32_t row_index_type;
  int64_t shared_rows;
  int64_t shared_offset;
  float shared_weight;
  uint32_t flags;
  int64_t expected_tokens_per_expert;
} gmmfr_problem;

/*
 * Bytes of the prepared-weight buffer for this problem's x2 and scale
 * (E x ceil(N/128) x ceil(K/128) tiles of 16896 bytes; packed E2M1 x1 and x2 with
 * K % 32 == 0: E x ceil(N/128) x ceil(K/256) tiles of 17408 bytes).  Host only; no CUDA call.
 * Returns GMMFR_ERR_INVALID_ARG on an invalid problem.
 */
GMMFR_API gmmfr_status gmmfr_prepared_weights_size(const gmmfr_problem* problem, size_t* bytes);

/*
 * One-time weight preparation: re-lays x2 and its E8M0 scale into the tiled,
 * swizzled layout the grouped GEMM streams (one 128-column x 128-K tile of FP8
 * weights followed by its 512 scale bytes), so that each tile is a single
 * contiguous HBM read.  Inputs as in section 3.1 (x2 [E,K,N] or [E,N,K]; scale
 * [(E,)ceil(K/64),N,2] or [(E,)N,ceil(K/64),2]); an E2M1 x2 is packed two codes
 * per byte along its last dimension.  With E2M1 tokens too (and K % 32 == 0) a tile
 * keeps the codes packed: 128 columns x 256 K (K pairs per byte, the lower K in the low
 * nibble) and then 1024 scale bytes (eight per row, in two 512-byte halves); otherwise
 * the E2M1 codes are stored prepared as E4M3 codes.
 *   x2, scale       views with the shapes above (checked as for the operator)
 *   prepared        device buffer of at least gmmfr_prepared_weights_size bytes,
 *                   16-byte aligned, caller-owned; fully overwritten.
 * Enqueued on `stream`; the buffer stays valid as long as the caller keeps it.
 */
GMMFR_API gmmfr_status gmmfr_prepare_weights(const gmmfr_problem* problem, const gmmfr_tensor* x2,
                                             const gmmfr_tensor* scale, void* prepared, size_t prepared_bytes,
                                             void* stream);

/*
 * Workspace bytes one call needs (two-phase use as in aclnn's
 * GetWorkspaceSize/execute pair).  `have_prepared` = 0 adds room to prepare
 * the weights inside the call; an E2M1 x1 that is expanded (x2 not E2M1, or
 * K % 32 != 0) adds M*K bytes for its expansion to E4M3, and x1 rows whose K is not a
 * multiple of 16 add M*Kp bytes (Kp = K rounded up to 16) for a copy at a 16-byte pitch
 * (the tensor copies that feed the GEMM need one).  Host only.  The workspace must be
 * 256-byte aligned.
 */
GMMFR_API gmmfr_status gmmfr_workspace_size(const gmmfr_problem* problem, int have_prepared, size_t* bytes);

/*
 * The operator.  Enqueues the whole computation on `stream`; never syncs and
 * never allocates.  Every view is checked against the problem first: a tensor of the wrong
 * rank, shape or element type, a layout that is not dense row-major, a missing required
 * tensor, or a buffer smaller than its stated size is refused with GMMFR_ERR_INVALID_ARG
 * (GMMFR_ERR_WORKSPACE for `prepared` and `workspace`) and nothing is enqueued.
 *   x1              [M,K] FP8 (E4M3 / E5M2 per x1_format; E2M1: [M,K/2] E2M1X2), required
 *                   when M > 0; 16-byte aligned when the GEMM reads it in place (FP8 codes,
 *                   or E2M1 tokens and weights kept packed, with K % 16 == 0)
 *   x2, scale       raw weights [E,K,N] / [E,N,K] and scales [(E,)ceil(K/64),N,2] /
 *                   [(E,)N,ceil(K/64),2] (E8M0); read only when prepared == NULL (they are
 *                   then prepared into the workspace first), and may be NULL otherwise
 *   pertoken_scale  [M,ceil(K/64),2] E8M0, required when M > 0
 *   group_list      [E] int64 (type per problem.group_list_type); values checked on the device
 *   logit           [M] float32, or NULL for weight 1 (has_logit = False)
 *   row_index       [M] int64 or int32 (problem.row_index_type), required when M > 0;
 *                   values in [0,batch), checked on the device
 *   shared_input    [shared_rows,N] bfloat16, required when shared_rows > 0
 *   bias            [E,N] bfloat16 (aclnn V3 biasOptional, BF16 on the MX path), or NULL;
 *                   read as a per-expert, per-column term added to the matmul result
 *                   before the logit weighting: out[r,n] += logit * (mm(t,n) + bias[e,n])
 *   out             [batch,N] float32, read and accumulated into in place
 *   prepared        output of gmmfr_prepare_weights for the same x2/scale (prepared_bytes of
 *                   it, at least gmmfr_prepared_weights_size), or NULL
 *   workspace       at least gmmfr_workspace_size bytes, 256-byte aligned; its
 *                   contents on entry do not matter; it must not be shared by two
 *                   calls in flight at the same time
 * Without GMMFR_DETERMINISTIC the row scatter uses float atomics, so the FP32
 * rounding order, and the low bits of `out`, can differ run to run (the aclnn
 * operator is non-deterministic by default, "确定性计算").  With it, every out
 * element is  ((out + c_t1) + c_t2) + ... + shared  over its tokens in
 * ascending order, and results are bit-identical run to run on one device.
 * Device-side index errors do not fail the call: they set bits of the device
 * error word, read with gmmfr_check_device_errors.
 * The grouped GEMM is launched as a programmatic dependent of the previous kernel in
 * `stream`: when that kernel allows it (gmmfr_moe_route does), the GEMM's launch
 * overlaps its tail; the GEMM reads no input before that kernel has completed.
 * Kernels per call: the grouped GEMM alone in the default mode; with
 * GMMFR_DETERMINISTIC the GEMM (which also builds the row CSR of the tokens) and then
 * the combine, a programmatic dependent of the GEMM.  Weights prepared inside the call
 * add the preparation kernel first, and an expanded E2M1 x1 the expansion kernel (or,
 * when K % 16 != 0, the copy of x1 to a 16-byte pitch, which also expands E2M1 codes).
 */
GMMFR_API gmmfr_status gmmfr_grouped_matmul_finalize_routing(
    const gmmfr_problem* problem, const gmmfr_tensor* x1, const gmmfr_tensor* x2, const gmmfr_tensor* scale,
    const gmmfr_tensor* pertoken_scale, const gmmfr_tensor* group_list, const gmmfr_tensor* logit,
    const gmmfr_tensor* row_index, const gmmfr_tensor* shared_input, const gmmfr_tensor* bias,
    const gmmfr_tensor* out, const void* prepared, size_t prepared_bytes, void* workspace, size_t workspace_bytes,
    void* stream);

/*
 * SYNCHRONISES `stream`, then reads the device error word that the last call
 * using `workspace` left there (GMMFR_DEV_* bits, 0 when clean) into *bits.
 * Returns GMMFR_ERR_DEVICE when any bit is set, GMMFR_OK otherwise.
 */
GMMFR_API gmmfr_status gmmfr_check_device_errors(const void* workspace, void* stream, uint32_t* bits);

/*
 * Allocation-free form of gmmfr_grouped_matmul_finalize_routing (no counterpart on
 * the source pages; added for callers that must not allocate device memory).
 *
 * Some callers cannot hand us a workspace: code embedded in a host runtime whose
 * memory pool owns the whole device and forbids outside allocations, serving
 * loops where a cudaMalloc (which can synchronise the device and fail under
 * memory pressure) is not acceptable, or plain C callers without an allocator.
 * This call takes the same tensors as the operator minus x2, scale, bias and the
 * workspace, and uses instead a 16 MiB scratch array compiled into the library
 * as a file-scope __device__ variable.  Every GPU that loads the library holds
 * those 16 MiB until the process exits.  It calls no cudaMalloc / cudaFree.
 *
 *   prepared   required: weights from gmmfr_prepare_weights (the call cannot prepare
 *              them itself), prepared_bytes of them; other arguments as for the operator
 *              (views, checked the same way).
 * Problems whose workspace (gmmfr_workspace_size with have_prepared = 1) exceeds
 * 16 MiB are rejected with GMMFR_ERR_WORKSPACE and a message giving both sizes.
 * Outside stream capture each call looks up the array's device address on the current
 * device (cudaGetSymbolAddress, with that device current), so the address stays right
 * after the device's context is destroyed and re-created.  Inside a capture the address
 * found by an earlier call on the device is used: make one call on each device before
 * any stream capture; a first call inside a capture returns GMMFR_ERR_UNSUPPORTED.
 * All calls share the one array and it keeps the last call's contents (the operator
 * rewrites every word it reads, so nothing needs clearing); calls that can overlap on
 * the GPU (different streams, or several host threads) race on it and must be
 * serialised by the caller.
 */
GMMFR_API gmmfr_status gmmfr_grouped_matmul_finalize_routing_static_scratch(
    const gmmfr_problem* problem, const gmmfr_tensor* x1, const gmmfr_tensor* pertoken_scale,
    const gmmfr_tensor* group_list, const gmmfr_tensor* logit, const gmmfr_tensor* row_index,
    const gmmfr_tensor* shared_input, const gmmfr_tensor* out, const void* prepared, size_t prepared_bytes,
    void* stream);

/*
 * gmmfr_check_device_errors for the allocation-free entry point: SYNCHRONISES `stream`,
 * then reads the device error word that the last static-scratch call on the current
 * device left in the library's scratch array (GMMFR_DEV_* bits) into *bits.  Returns
 * GMMFR_ERR_DEVICE when any bit is set, GMMFR_OK otherwise.
 */
GMMFR_API gmmfr_status gmmfr_static_scratch_check_device_errors(void* stream, uint32_t* bits);

/*
 * The routing step before the operator (LLaDA2.0-mini grouped-GEMM write-up,
 * section 5.2: argsort of the flattened expert ids, bincount, cumsum, and the
 * tokens gathered in that order).  It produces the operator's x1,
 * pertoken_scale, group_list, row_index and logit from tokens that are not yet
 * routed and their top-k expert choice.
 *
 *   batch, topk   tokens and experts per token; M = batch * topk routed entries
 *   K, E          row length of x (any K >= 1) and number of experts (1..1024)
 *   ids_type      gmmfr_index_type of topk_ids
 *   group_list_type  format of the produced group_list (0 prefix sums, 1 counts)
 */
typedef struct {
  int64_t batch, topk, K, E;
  int32_t ids_type;
  int32_t group_list_type;
} gmmfr_route_problem;

/* Workspace bytes of gmmfr_moe_route (256-byte aligned).  Host only. */
GMMFR_API gmmfr_status gmmfr_moe_route_workspace_size(const gmmfr_route_problem* problem, size_t* bytes);

/*
 * Entry f = b * topk + k (expert topk_ids[b, k]) goes to output position
 *   (number of entries with a smaller expert id) + (entries of the same expert with a smaller f),
 * i.e. a stable sort by expert; entries whose id lies outside [0, E) are placed
 * after every routed entry (in ascending f), belong to no group, and set
 * GMMFR_DEV_BAD_EXPERT_ID in the device error word of `workspace`.  At position p
 * holding entry f:  x1[p] = x[f / topk], pertoken_scale[p] = x_scale[f / topk],
 * row_index[p] = f / topk, logit[p] = topk_weights[f] (1 when topk_weights is NULL),
 * perm[p] = f.
 *   inputs   topk_ids [batch, topk]; topk_weights [batch, topk] float32 or NULL;
 *            x [batch, K] FP8 bytes; x_scale [batch, ceil(K/64), 2] E8M0 bytes
 *   outputs  x1 [M, K]; pertoken_scale [M, ceil(K/64), 2]; group_list [E] int64;
 *            row_index [M] int64; logit [M] float32 or NULL; perm [M] int32 or NULL
 * One kernel launch up to 8192 entries (M), three above; never syncs, never allocates.
 * Bit-exact and deterministic (byte and index work only).
 */
GMMFR_API gmmfr_status gmmfr_moe_route(const gmmfr_route_problem* problem, const void* topk_ids,
                                       const float* topk_weights, const void* x, const void* x_scale, void* x1,
                                       void* pertoken_scale, int64_t* group_list, int64_t* row_index, float* logit,
                                       int32_t* perm, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Grouped SwiGLU expert FFN in BF16 (llada2_moe_grouped_gemm; LLaDA2.0-mini
 * grouped-GEMM write-up, sections 3.1-3.3).  For every expert e and its sorted
 * token rows [expert_cumsum[e], expert_cumsum[e+1]):
 *   gate_up = x @ w13_flat[e*H:(e+1)*H, :]   (FP32 accumulate; gate = first I columns, up = last I)
 *   sw      = bf16(SiLU(gate) * up),  SiLU(g) = g / (1 + exp(-g))
 *   result  = bf16(sw @ w2_flat[e*I:(e+1)*I, :])
 * Rows outside every expert range are left untouched.
 *   N  rows of sorted_tokens and result;  H, I  hidden and intermediate sizes
 *      (multiples of 8);  E  experts (1..1024)
 */
typedef struct {
  int64_t N, H, I, E;
} gmmfr_ffn_problem;

/* Bytes of the prepared FFN weights (E*ceil(I/64)*ceil(H/64) + E*ceil(H/128)*ceil(I/64) tiles of 16 KB). */
GMMFR_API gmmfr_status gmmfr_ffn_prepared_weights_size(const gmmfr_ffn_problem* problem, size_t* bytes);

/* One-time re-layout of w13_flat [E*H, 2I] and w2_flat [E*I, H] (bf16) into swizzled
 * 128-row tiles (a w13 tile holds 64 gate columns and the 64 up columns of the same
 * indices); `prepared` is a caller buffer, 16-byte aligned, fully overwritten. */
GMMFR_API gmmfr_status gmmfr_ffn_prepare_weights(const gmmfr_ffn_problem* problem, const void* w13_flat,
                                                 const void* w2_flat, void* prepared, size_t prepared_bytes,
                                                 void* stream);

/* Workspace bytes of gmmfr_llada2_moe_grouped_gemm (error words + the bf16 sw rows). */
GMMFR_API gmmfr_status gmmfr_ffn_workspace_size(const gmmfr_ffn_problem* problem, size_t* bytes);

/* The grouped FFN: sorted_tokens [N, H] bf16, expert_cumsum [E+1] int32 (checked on the
 * device: non-decreasing, within [0, N]; violations set GMMFR_DEV_BAD_GROUP_LIST and are
 * clamped), result [N, H] bf16.  Two kernel launches; no sync, no allocation; every
 * result element is written by one thread (deterministic). */
GMMFR_API gmmfr_status gmmfr_llada2_moe_grouped_gemm(const gmmfr_ffn_problem* problem, const void* sorted_tokens,
                                                     const void* prepared, const int32_t* expert_cumsum,
                                                     void* result, void* workspace, size_t workspace_bytes,
                                                     void* stream);

/* Message of the last error returned on the calling thread ("" if none). */
GMMFR_API const char* gmmfr_last_error(void);

/*
 * Kernel timing for measurement.  gmmfr_profile_begin(n) creates CUDA events
 * for up to n calls; each later call records events around each of its
 * kernels on its stream.  gmmfr_profile_end SYNCHRONISES the device, writes
 * ms[call * GMMFR_PROFILE_SLOTS + slot] (-1 where a slot's kernel did not run),
 * sets *n_calls, and stops recording.
 * Slots: 0 input preparation inside the call (weight preparation when no prepared
 * weights are given, E2M1 token expansion), 1 not used (the deterministic mode's
 * row CSR of the tokens is built inside the grouped GEMM), 2 grouped GEMM with fused
 * epilogue, 3 deterministic combine, 4 the whole call (start of its first kernel to
 * end of its last).
 */
#define GMMFR_PROFILE_SLOTS 5
GMMFR_API gmmfr_status gmmfr_profile_begin(int max_calls);
GMMFR_API gmmfr_status gmmfr_profile_end(float* ms, int max_entries, int* n_calls);

#ifdef __cplusplus
}
#endif
#endif /* GMMFR_H */
