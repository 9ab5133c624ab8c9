/*
 * moe_a16w4.h - C ABI of the GB300 (sm_103a) A16W4 mixture-of-experts library.
 *
 * The layer: BF16 activations, MXFP4 expert weights (packed E2M1 nibbles, two per
 * byte, one E8M0 scale byte per 32 elements along K), SiLU-gated MLP experts,
 * top-k weighted combine.  Source: the vLLM ``Mxfp4MoEMethod`` API page
 * (quantization/mxfp4): ``create_weights`` fixes the weight layouts used below,
 * ``apply`` the forward call, ``_setup_kernel_k3_situ_gfx942`` the opt-in
 * MXFP4 -> int4_per_group_32 requantisation; vLLM PR #51274 (Summary, Changes)
 * the lossy opt-in int4 path and its eight-experts-per-chunk conversion.
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

/* Activation selector.  Only the SiLU-gated one the pages' stage-1 kernels
 * compute is implemented; SiTUv2 is named on the pages without a formula. */
#define MOE_ACT_SWIGLU 0

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
 * (0 if ``d`` is invalid).  The caller allocates it (256-byte aligned) and may
 * reuse it across calls that are ordered on one stream; calls that can run
 * concurrently need separate workspaces.  The outputs do not depend on what the
 * workspace held before: the words the kernels synchronise through carry a
 * per-call value that leftovers do not match.  Only the status word (its
 * first 4 bytes) reads back what the memory held until it is first cleared:
 * zero those bytes, or call moe_read_status once, after allocating. */
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
 * Same layer on int4_per_group_32 weights (the requantiser's output format):
 *   w13_q  uint8 [E, 2I, H/2]  two's-complement int4, element 2j low    16-byte aligned
 *   w13_s  float32 [E, 2I, H/32] one scale per 32-group                  16-byte aligned
 *   w2_q   uint8 [E, H, I/2],  w2_s float32 [E, H, I/32]                 16-byte aligned
 * Weight value = q * s.  The weight-streaming kernels apply s to each group's
 * partial sum in fp32; the tensor-core kernels (large batches, same rules as
 * moe_a16w4_mxfp4 for ``d->path``) multiply with bf16(fl32(q * s)).
 */
int moe_a16w4_int4g32(const moe_dims_t* d, const void* x, const int32_t* topk_ids,
                      const float* topk_w, const uint8_t* w13_q, const float* w13_s,
                      const uint8_t* w2_q, const float* w2_s, void* out, void* workspace,
                      size_t workspace_bytes, void* stream);

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
 * Source and destination must not overlap.  Scale bytes of 255 (NaN) are
 * outside the contract.  K multiple of 32, N >= 1, E >= 1.
 */
int requant_mxfp4_to_int4g32(int32_t E, int32_t N, int32_t K, const uint8_t* w, const uint8_t* scale,
                             uint8_t* out_q, float* out_s, int32_t experts_per_chunk, void* stream);

/*
 * The grouping step alone (stable counting sort of the T*topk pairs by expert):
 *   counts      int32 [E]     pairs per expert
 *   offsets     int32 [E+1]   exclusive prefix sum of counts
 *   sorted_pair int32 [T*topk] flat pair index t*topk+k, ascending within each
 *               expert; entries from offsets[E] on are -1
 *   pair_pos    int32 [T*topk] position of each pair in sorted_pair, -1 if its id is invalid
 * Only d->E, d->topk and d->T are read.
 */
int moe_route(const moe_dims_t* d, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
              int32_t* sorted_pair, int32_t* pair_pos, void* stream);

/* Copy the device status word of ``workspace`` (MOE_STATUS_* bits, 0 = clean)
 * into *status and clear it, together with the words the decode kernels
 * synchronise through (after a wait that gave up, those may be inconsistent;
 * read the status before reusing such a workspace).  Synchronises ``stream``. */
int moe_read_status(const moe_dims_t* d, void* workspace, uint32_t* status, void* stream);

/*
 * Allocation-free variant of moe_a16w4_mxfp4.  The pages have no counterpart:
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
 *   - All calls share the one array, which keeps the previous call's contents;
 *     every region is written before it is read within a call, so nothing needs
 *     clearing.  Calls that may overlap on the GPU (different streams, or
 *     different host threads on one device) race on the array: order them.
 *   - Device status bits of this variant are not exposed.
 */
int moe_a16w4_mxfp4_noalloc(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2,
                            const uint8_t* w2_scale, void* out, void* stream);

/*
 * Optional per-kernel timing, for benchmarks.  ``events`` holds 2*n
 * cudaEvent_t handles created by the caller (n <= 8).  The next
 * moe_a16w4_mxfp4 / moe_a16w4_int4g32 call made from this host thread records
 * events[2i] just before and events[2i+1] just after its i-th kernel launch
 * (i < n) on the call's stream; the hook is then cleared.  Kernel order:
 * weight-streaming path 0 grouping, 1 gate_up GEMM, 2 down GEMM, 3 combine,
 * where H and I are at most 3584 one launch runs both GEMMs (index 1) and
 * the index-2 events are recorded back to back; tensor-core path 0 grouping,
 * 1 row gather, 2 gate_up GEMM, 3 down GEMM, 4 combine.  Slots without a
 * launch (grouping of at most 128 pairs, done inside the decode kernels) are
 * recorded back to back too.  n = 0 clears the hook.  Returns
 * MOE_ERR_BAD_DIMS for n outside [0, 8] and MOE_ERR_NULL for a NULL
 * ``events`` with n > 0.
 */
int moe_set_timing_events(void* const* events, int32_t n);

/* Static text for a MOE_ERR_* code. */
const char* moe_error_string(int code);

/* Library ABI version (major*100 + minor). */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_A16W4_H */
