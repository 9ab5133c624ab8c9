/*
 * moe_a16w4.h - C ABI of the GB300 (sm_103a) A16W4 mixture-of-experts library.
 *
 * The layer: BF16 activations, MXFP4 expert weights (packed E2M1 nibbles, two per
 * byte, one E8M0 scale byte per 32 elements along K), SiLU-gated MLP experts,
 * top-k weighted combine.  Source: the vLLM ``Mxfp4MoEMethod`` API page
 * (quantization/mxfp4): ``create_weights`` fixes the weight layouts used below,
 * ``apply`` the forward call, ``_setup_kernel_k3_situ_gfx942`` the opt-in
 * MXFP4 -> int4_per_group_32 requantisation; vLLM PR #51274 (Summary, Changes)
 * the lossy opt-in int4 path and its eight-experts-per-chunk conversion (with
 * float32 or, per its commit message, bf16 group scales); vLLM PR #39136 the
 * W4A4 / W4A8 schemes (quantised activations, moe_options_t.act_quant).
 * The same sources built with -DMOE_CHECK give libmoe_a16w4_check.so, the
 * bounds-checked build (MOE_STATUS_BAD_INDEX, MOE_STATUS_NAN_SCALE).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers to caller-owned memory, dense and
 *    row-major (C order).  The library never allocates, frees or synchronises
 *    the host; work is enqueued on ``stream`` (a cudaStream_t, NULL = legacy
 *    default stream) and the call returns before it finishes.
 *  - bf16 tensors are passed as ``const void*`` / ``void*`` holding IEEE
 *    bfloat16 bit patterns.
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  Argument checks
 *    happen before any CUDA call; when one fails nothing is enqueued.
 *  - Device-side problems that cannot be seen on the host (a bounded wait in a
 *    kernel that ran out) are recorded in a status word inside the workspace;
 *    read and clear it with moe_read_status().
 */
#ifndef MOE_A16W4_H
#define MOE_A16W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_NULL (-1)            /* a required pointer is NULL                          */
#define MOE_ERR_BAD_DIMS (-2)        /* sizes outside the supported set (see moe_dims_t)    */
#define MOE_ERR_ALIGN (-3)           /* a pointer is not aligned as documented              */
#define MOE_ERR_UNSUPPORTED_ACT (-4) /* activation other than SwiGLU: fail closed            */
#define MOE_ERR_WORKSPACE (-5)       /* workspace smaller than moe_workspace_bytes()         */
#define MOE_ERR_CUDA (-6)            /* a CUDA runtime call or launch failed                 */
#define MOE_ERR_DEVICE (-7)          /* current device is not a compute capability 10.3 GPU  */

/* Device status bits (moe_read_status). */
#define MOE_STATUS_WAIT_TIMEOUT 0x1u /* a pipeline wait in a kernel gave up; outputs invalid */
/* Set only by the checked build of the library (libmoe_a16w4_check.so, the
 * same sources compiled with -DMOE_CHECK), whose kernels check every index
 * they derive (expert, pair, token, row, tile) against its buffer and every
 * E8M0 weight-scale byte they read -- a stand-in for a memory checker: */
#define MOE_STATUS_BAD_INDEX 0x2u    /* an index was out of range; it was replaced by 0 (outputs invalid) */
#define MOE_STATUS_NAN_SCALE 0x4u    /* an E8M0 weight-scale byte was 255 (NaN in the format)          */

/* Activation selector.  Only the SiLU-gated one the pages' stage-1 kernels
 * compute is implemented; SiTUv2 is named on the pages without a formula. */
#define MOE_ACT_SWIGLU 0

/* Activation quantisation of both GEMM inputs (moe_options_t.act_quant):
 * the OCP MX schemes of vLLM PR #39136 ("[ROCm][Quantization][2/N] Refactor
 * quark_moe w4a8 w/ oracle", Summary and review): ``w_mxfp4_a_mxfp4`` (W4A4)
 * and ``w_mxfp4_a_fp8`` (W4A8, static FP8 activations). */
#define MOE_AQ_NONE 0  /* bf16 activations (the A16W4 layer)                              */
#define MOE_AQ_MXFP4 1 /* MXFP4 activations: E2M1 + E8M0 per 32 values along K           */
#define MOE_AQ_FP8 2   /* e4m3fn activations with one static float32 scale per GEMM input */

/* Kernel family selector (moe_dims_t.path). */
#define MOE_PATH_AUTO 0    /* weight-streaming kernels for small batches, tensor-core kernels for large */
#define MOE_PATH_DECODE 1  /* force the weight-streaming (decode) kernels                              */
#define MOE_PATH_PREFILL 2 /* force the tcgen05 tensor-core (prefill) kernels                          */

/*
 * Problem size of one MoE layer call.
 *   E     experts held by this GPU (ids 0..E-1)            1 <= E <= 1024
 *   H     hidden size (K of the gate_up GEMM)              multiple of 64, 64 <= H <= 4096
 *   I     intermediate size per expert (K of the down GEMM) multiple of 64, 64 <= I <= 4096
 *   topk  experts per token                                1 <= topk <= 64
 *   T     tokens                                           0 <= T, T*topk <= 2^24
 *   act   MOE_ACT_SWIGLU
 *   path  MOE_PATH_*; the tensor-core path additionally needs H and I to be
 *         multiples of 512 (MOE_PATH_AUTO falls back to the weight-streaming
 *         kernels otherwise)
 */
typedef struct moe_dims {
  int32_t E, H, I, topk, T;
  int32_t act;
  int32_t path;
} moe_dims_t;

/* Bytes of scratch that moe_a16w4_mxfp4 / moe_a16w4_int4g32 need for ``d``
 * (0 if ``d`` is invalid).  Source: vLLM PR #51274, Validation -- the layer
 * runs under full and piecewise CUDA graph capture, so a call may not
 * allocate; the caller allocates this scratch once (256-byte aligned) and
 * passes it to every call.  It may be reused across calls that are ordered on
 * one stream; calls that can run concurrently need separate workspaces.  The
 * outputs do not depend on what the workspace held before: the words the
 * kernels synchronise through carry a per-call value that leftovers do not
 * match.  Only the status word (its first 4 bytes) reads back what the memory
 * held until it is first cleared: zero those bytes, or call moe_read_status
 * once, after allocating. */
size_t moe_workspace_bytes(const moe_dims_t* d);

/*
 * Fused MoE forward, MXFP4 weights (Mxfp4MoEMethod.apply semantics, W4A16:
 * weights dequantised, activations kept BF16, fp32 accumulation).
 *   x          bf16 [T, H]                       16-byte aligned
 *   topk_ids   int32 [T, topk]; ids outside [0, E) contribute nothing
 *   topk_w     float32 [T, topk]
 *   w13        uint8 [E, 2I, H/2]  E2M1 pairs, element 2j in the low nibble;
 *              rows [0, I) gate, rows [I, 2I) up           16-byte aligned
 *   w13_scale  uint8 [E, 2I, H/32] E8M0, value 2^(s-127)   16-byte aligned
 *   w2         uint8 [E, H, I/2]                           16-byte aligned
 *   w2_scale   uint8 [E, H, I/32]                          16-byte aligned
 *   out        bf16 [T, H], fully overwritten               16-byte aligned
 *   out[t] = sum_k topk_w[t,k] * W2[e] (SiLU(W13[e][:I] x[t]) * (W13[e][I:] x[t])),
 *   e = topk_ids[t,k], summed in k order, rounded to bf16 once.
 */
int moe_a16w4_mxfp4(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                    const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                    const uint8_t* w2_scale, void* out, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Same layer on int4_per_group_32 weights (the requantiser's output format).
 * Source: vLLM PR #51274, Summary -- the opt-in int4_per_group_32 MoE path
 * serves the requantised experts through a BF16 x packed-int4 kernel; the
 * Mxfp4MoEMethod page's _setup_kernel_k3_situ_gfx942 hands that kernel the
 * converted w13/w2 and their per-32-group scales in place of the MXFP4 ones.
 *   w13_q  uint8 [E, 2I, H/2]  two's-complement int4, element 2j low    16-byte aligned
 *   w13_s  float32 [E, 2I, H/32] one scale per 32-group                  16-byte aligned
 *   w2_q   uint8 [E, H, I/2],  w2_s float32 [E, H, I/32]                 16-byte aligned
 * Weight value = q * s.  The weight-streaming kernels apply s to each group's
 * partial sum in fp32; the tensor-core kernels (large batches, same rules as
 * moe_a16w4_mxfp4 for ``d->path``) multiply with bf16(fl32(q * s)) in the
 * gate_up GEMM and f16(q * f16(s * 2^ew)) in the down GEMM (ew a power of
 * two per weight row that puts the row's largest weight just below 2^15).
 */
int moe_a16w4_int4g32(const moe_dims_t* d, const void* x, const int32_t* topk_ids,
                      const float* topk_w, const uint8_t* w13_q, const float* w13_s,
                      const uint8_t* w2_q, const float* w2_s, void* out, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Optional inputs of the layer call.  Source: the Mxfp4MoEMethod page --
 * ``create_weights`` registers ``w13_bias`` bf16 [E, 2I] and ``w2_bias``
 * bf16 [E, H] when the layer has biases and ``get_fused_moe_quant_config``
 * hands them to the kernel (``w1_bias``, ``w2_bias``); ``apply`` passes
 * ``global_num_experts``, ``expert_map`` and ``apply_router_weight_on_input``.
 * The pages print no formula for any of them; the readings used:
 *   w13_bias               added to the gate_up GEMM's outputs before the
 *                          activation: h = W13[e] x + b13[e]
 *   w2_bias                added to each expert's output: y = W2[e] a + b2[e]
 *   router_weight_on_input each pair's input is scaled by its router weight
 *                          (h = W13[e] (w x) + b13[e]) and the combine sums the
 *                          pairs' outputs unweighted
 *   expert_map             topk_ids hold global expert ids in
 *                          [0, global_num_experts); expert_map[g] is the local
 *                          id (0..E-1) of global expert g, or -1 if another GPU
 *                          holds it; ids outside the map or mapped to -1
 *                          contribute nothing
 * Activation quantisation (MOE_AQ_*; MXFP4 weights only, and not together
 * with router_weight_on_input): each GEMM's input -- x for gate_up, the
 * SiLU-gated intermediate a (float32 in the kernels) for down -- is replaced
 * by its quantised-dequantised value, as moe_quantize_act() defines it
 * (MXFP4 per 32-value block of each row; FP8 with w13_input_scale for x and
 * w2_input_scale for a).  The GEMMs run on exact codes (FP8: the e4m3 values,
 * the scale applied to the float32 result).
 * swiglu_limit: ``get_fused_moe_quant_config`` passes the layer's
 * ``swiglu_limit`` as ``gemm1_clamp_limit``, without a formula; reading used:
 * the gate_up GEMM's output, bias included, clamped element by element to
 * [-limit, limit] before the SiLU gating (h = clamp(W13[e] x + b13[e])).
 * A zero-initialised struct (all NULL / 0) is the plain layer.
 */
typedef struct moe_options {
  const void* w13_bias;            /* bf16 [E, 2I] or NULL (2-byte aligned) */
  const void* w2_bias;             /* bf16 [E, H] or NULL (2-byte aligned)  */
  const int32_t* expert_map;       /* int32 [global_num_experts] or NULL    */
  int32_t global_num_experts;      /* 1 .. 2^20 when expert_map is set      */
  int32_t router_weight_on_input;  /* 0 or 1                                */
  int32_t act_quant;               /* MOE_AQ_*                              */
  float w13_input_scale;           /* MOE_AQ_FP8: finite, > 0               */
  float w2_input_scale;            /* MOE_AQ_FP8: finite, > 0               */
  float swiglu_limit;              /* 0: off; else finite, > 0              */
} moe_options_t;

/* moe_a16w4_mxfp4 / moe_a16w4_int4g32 with optional inputs (``opt`` may be
 * NULL: the plain call).  Returns MOE_ERR_BAD_DIMS for global_num_experts
 * outside [1, 2^20] with a map, router_weight_on_input not 0 or 1, act_quant
 * outside MOE_AQ_*, an FP8 input scale that is not finite and positive, a
 * swiglu_limit that is negative, infinite or NaN, or act_quant set with int4
 * weights or with router_weight_on_input. */
int moe_a16w4_mxfp4_ex(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                       const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                       const uint8_t* w2_scale, const moe_options_t* opt, void* out, void* workspace,
                       size_t workspace_bytes, void* stream);
int moe_a16w4_int4g32_ex(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                         const uint8_t* w13_q, const float* w13_s, const uint8_t* w2_q, const float* w2_s,
                         const moe_options_t* opt, void* out, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Load-time, lossy MXFP4 -> int4_per_group_32 requantisation
 * (_setup_kernel_k3_situ_gfx942's convert(): decode E2M1 and E8M0, scale each
 * 32-block, cast to bf16 (exact for these values), then symmetric int4 per
 * 32-group: scale = fl32(amax / 7), q = round-half-even(fl32(w / scale)),
 * clamped to [-8, 7]; an all-zero group gets scale 0 and q 0).
 *   w      uint8 [E, N, K/2]   MXFP4 elements     16-byte aligned
 *   scale  uint8 [E, N, K/32]  E8M0
 *   out_q  uint8 [E, N, K/2]   int4 pairs, element 2j low   16-byte aligned
 *   out_s  float32 [E, N, K/32]                              16-byte aligned
 * Experts are converted ``experts_per_chunk`` at a time (one launch per
 * chunk; 8 on the pages); the result does not depend on the chunk size.
 * Source and destination must not overlap.  Results are bit-exact for scale
 * bytes 0..252; bytes 253 and 254 are outside the contract (E2M1 codes 4 and 6
 * times 2^126 or 2^127 overflow float32) and so is 255 (NaN).  K multiple of
 * 32, N >= 1, E >= 1.
 */
int requant_mxfp4_to_int4g32(int32_t E, int32_t N, int32_t K, const uint8_t* w, const uint8_t* scale,
                             uint8_t* out_q, float* out_s, int32_t experts_per_chunk, void* stream);

/*
 * int4_per_group_32 with bfloat16 group scales.  Source: vLLM PR #51274,
 * commit message -- the MXFP4 expert weights are converted "to int4 with
 * groupwise bf16 scales" (the float32-scale calls above follow the other
 * reading).  Reading used: the scale fl32(amax / 7) is rounded to bf16
 * (nearest even) and the elements are quantised against that stored scale,
 * q = round-half-even(fl32(w / scale_bf16)) in [-8, 7] (never -8 in fact).
 *   requant_mxfp4_to_int4g32_bf16s: as requant_mxfp4_to_int4g32 with
 *     out_s bf16 [E, N, K/32] (16-byte aligned); bit-exact for scale bytes
 *     0..252.
 *   moe_a16w4_int4g32_bf16s(_ex): as moe_a16w4_int4g32(_ex) with
 *     w13_s bf16 [E, 2I, H/32] and w2_s bf16 [E, H, I/32] (16-byte aligned);
 *     weight value q * s.  act_quant is rejected as for float32 scales.
 */
int requant_mxfp4_to_int4g32_bf16s(int32_t E, int32_t N, int32_t K, const uint8_t* w, const uint8_t* scale,
                                   uint8_t* out_q, void* out_s, int32_t experts_per_chunk, void* stream);
int moe_a16w4_int4g32_bf16s(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13_q, const void* w13_s, const uint8_t* w2_q, const void* w2_s,
                            void* out, void* workspace, size_t workspace_bytes, void* stream);
int moe_a16w4_int4g32_bf16s_ex(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                               const uint8_t* w13_q, const void* w13_s, const uint8_t* w2_q, const void* w2_s,
                               const moe_options_t* opt, void* out, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * The grouping step alone.  Source: the Mxfp4MoEMethod page, ``apply`` -- the
 * fused-MoE kernel receives topk_ids and topk_weights [T, topk] (ids of
 * non-local experts arrive as -1 through ``expert_map``) and must bring each
 * expert's (token, slot) pairs together before its grouped GEMMs.  The pages
 * give no order; this is a stable counting sort of the T*topk pairs by expert:
 *   counts      int32 [E]     pairs per expert
 *   offsets     int32 [E+1]   exclusive prefix sum of counts
 *   sorted_pair int32 [T*topk] flat pair index t*topk+k, ascending within each
 *               expert; entries from offsets[E] on are -1
 *   pair_pos    int32 [T*topk] position of each pair in sorted_pair, -1 if its id is invalid
 * Only d->E, d->topk and d->T are read.
 */
int moe_route(const moe_dims_t* d, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
              int32_t* sorted_pair, int32_t* pair_pos, void* stream);

/*
 * Top-k routing from router logits.  Source: the Mxfp4MoEMethod page,
 * ``apply_monolithic`` -- the kernel receives ``router_logits`` instead of
 * top-k ids and weights and chooses the experts itself; the pages print no
 * scoring formula.  The plain reading implemented: p = softmax over each
 * token's logits; the ``topk`` largest p are kept (in decreasing order, ties
 * to the lower expert id); with ``renormalize`` the kept p are divided by
 * their sum.  Grouped top-k, a score-correction bias and a routed scaling
 * factor (named on the page) are not modelled.
 *   logits    float32 [T, G], G = experts seen by the router (global ids when
 *             the layer then maps them through moe_options_t.expert_map)
 *   topk_ids  int32 [T, topk]   (bit-exact: selection by logit, which orders
 *             the experts exactly as their probabilities do)
 *   topk_w    float32 [T, topk] (float32 exp and one IEEE division each)
 * 1 <= G <= 1024, 1 <= topk <= min(64, G), renormalize 0 or 1.  NaN logits
 * are outside the contract.
 */
int moe_router_topk(const float* logits, int32_t T, int32_t G, int32_t topk, int32_t renormalize,
                    int32_t* topk_ids, float* topk_w, void* stream);

/* Copy the device status word of ``workspace`` (MOE_STATUS_* bits, 0 = clean)
 * into *status and clear it, together with the words the decode kernels
 * synchronise through (after a wait that gave up, those may be inconsistent;
 * read the status before reusing such a workspace).  Synchronises ``stream``.
 * The pages have no counterpart: their kernels do not wait on one another.
 * The fail-closed principle of the Mxfp4MoEMethod page (an unsupported
 * activation is an error, never a silent substitute) is why a wait that ran
 * out is reported here rather than left as silently wrong output. */
int moe_read_status(const moe_dims_t* d, void* workspace, uint32_t* status, void* stream);

/*
 * Bounded-wait hook for the next moe_a16w4_mxfp4 / moe_a16w4_int4g32 call made
 * from this host thread (then cleared).  The pages have no counterpart.
 *   limit_ns       limit of every wait inside that call's kernels, instead of
 *                  the default 2 s; a wait that runs out sets
 *                  MOE_STATUS_WAIT_TIMEOUT, the kernels stop and return, and the
 *                  call's output is invalid (> 0)
 *   extra_waiters  for tests of the give-up path: the fused decode kernel's
 *                  wait for all of its CTAs' gate_up results expects this many
 *                  CTAs more than it launched, so that wait runs out after
 *                  limit_ns (0..64; 0 for normal use)
 * Returns MOE_ERR_BAD_DIMS for limit_ns = 0 or extra_waiters outside [0, 64].
 */
int moe_set_wait_limit(uint64_t limit_ns, int32_t extra_waiters);

/*
 * Allocation-free variant of moe_a16w4_mxfp4.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory when
 * they run the layer (a serving thread that must not call cudaMalloc or a
 * framework allocator, a plugin that is handed only input and output pointers,
 * a process whose device memory is reserved up front).  It takes the same
 * inputs and output as moe_a16w4_mxfp4 but no workspace: its scratch is one
 * fixed 16 MiB device array inside the library, which every GPU that loads the
 * library holds until the process exits.
 *   - Runs the weight-streaming kernels (d->path AUTO or DECODE; PREFILL is
 *     rejected with MOE_ERR_BAD_DIMS).  Problems whose workspace
 *     (moe_workspace_bytes with path DECODE) exceeds 16 MiB are rejected with
 *     MOE_ERR_WORKSPACE; the 112-expert, H=3584, I=3072, top-15 layer fits up
 *     to 32 tokens.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (once per device, with that device current); make
 *     that first call before any stream capture.
 *   - All calls share the one array, which keeps the previous call's contents.
 *     Its data regions are written before they are read within a call; its
 *     synchronisation words carry a per-call value that leftovers do not
 *     match, and the one kernel that synchronises through them is launched so
 *     that all of its CTAs run at once.  Calls that may overlap on the GPU
 *     (different streams, or different host threads on one device) race on the
 *     array: order them.
 *   - A bounded wait that ran out (MOE_STATUS_WAIT_TIMEOUT) is recorded in the
 *     array's status word: read and clear it with moe_noalloc_read_status.
 */
int moe_a16w4_mxfp4_noalloc(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                            const uint8_t* w2_scale, void* out, void* stream);

/* Status word of the current device's allocation-free scratch array (as
 * moe_read_status does for a workspace): copies it to *status and clears it
 * and the array's synchronisation words.  Synchronises ``stream``; allocates
 * nothing.  The paper has no counterpart. */
int moe_noalloc_read_status(uint32_t* status, void* stream);

/*
 * Optional per-kernel timing, for benchmarks.  ``events`` holds 2*n
 * cudaEvent_t handles created by the caller (n <= 8).  The next
 * moe_a16w4_mxfp4 / moe_a16w4_int4g32 call made from this host thread records
 * events[2i] just before and events[2i+1] just after its i-th kernel launch
 * (i < n) on the call's stream; the hook is then cleared.  Kernel order:
 * weight-streaming path 0 grouping, 1 gate_up GEMM, 2 down GEMM, 3 combine,
 * where H and I are at most 3584 one launch runs both GEMMs (index 1) and
 * the index-2 events are recorded back to back; tensor-core path 0 grouping,
 * 1 row gather, 2 gate_up GEMM, 3 f16 conversion of the intermediate, 4 down
 * GEMM (with the weighted combine), 5 bf16 cast of the output.  Slots without a
 * launch (grouping of at most 128 pairs, done inside the decode kernels) are
 * recorded back to back too.  n = 0 clears the hook.  Returns
 * MOE_ERR_BAD_DIMS for n outside [0, 8] and MOE_ERR_NULL for a NULL
 * ``events`` with n > 0.
 */
int moe_set_timing_events(void* const* events, int32_t n);

/*
 * Activation quantiser of the W4A4 / W4A8 schemes (vLLM PR #39136:
 * ``w_mxfp4_a_mxfp4``, ``w_mxfp4_a_fp8``; the pages name the schemes, the
 * rules below are the plain readings): the routine the layer kernels apply
 * to each GEMM input, as a call of its own.
 *   x          [rows, K] row-major, bf16 (x_is_f32 = 0) or float32 (1);
 *              16-byte aligned; finite values
 *   K          multiple of 32, 32 .. 2^20; rows 0 .. 2^31
 *   MOE_AQ_MXFP4: per 32 consecutive values of a row, the OCP MX v1.0 scale
 *              byte floor(log2 amax) - 2 + 127 (0 when amax < 2^-125, zero
 *              included) -> q_scale [rows, K/32]; each value times
 *              2^(127 - byte) rounded to the nearest E2M1 value, ties to the
 *              even code, saturating at +-6 -> q [rows, K/2] (value 2j in the
 *              low nibble of byte j); the sign bit follows the input.
 *   MOE_AQ_FP8: r = fl32(x / scale) (correctly rounded), rounded to the
 *              nearest e4m3fn value, ties to even, saturating at +-448 ->
 *              q [rows, K] (one code per byte); q_scale unused (may be NULL).
 *   q          16-byte aligned; caller-owned outputs, written on ``stream``.
 * Returns MOE_ERR_BAD_DIMS for a bad mode, dtype, size or FP8 scale,
 * MOE_ERR_NULL / MOE_ERR_ALIGN for the pointers.
 */
int moe_quantize_act(int32_t act_quant, const void* x, int32_t x_is_f32, int64_t rows, int32_t K, float scale,
                     uint8_t* q, uint8_t* q_scale, void* stream);

/* Static text for a MOE_ERR_* code. */
const char* moe_error_string(int code);

/* Library ABI version (major*100 + minor). */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_A16W4_H */
