// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_a16w4.h"

namespace moe {

constexpr uint32_t kStatusWaitTimeout = MOE_STATUS_WAIT_TIMEOUT;
constexpr uint32_t kStatusBadIndex = MOE_STATUS_BAD_INDEX;
constexpr uint32_t kStatusNanScale = MOE_STATUS_NAN_SCALE;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait

constexpr int kMaxExperts = 1024;
constexpr int kRouteThreads = 1024;

// Pairs per activation group of the weight-streaming kernels.
constexpr int kMoeGroup = 8;

// Pairs (tokens x topk) up to which the decode kernels group the pairs
// themselves and no routing kernel runs.
constexpr int kMaxLocalRoutePairs = 128;
// Tokens at or above which MOE_PATH_AUTO picks the tensor-core kernels.
constexpr int kPrefillMinTokens = 64;
// Whether the tensor-core (prefill) kernels are built into this library.
constexpr bool kPrefillAvailable = true;

// Prefill tile sizes (tcgen05, cta_group::1).  The MMA's M side is a tile of
// 128 dequantised weight rows held in tensor memory; its N side is a tile of
// up to kTcRowsUp (gate_up) or kTcRowsDown (down) sorted activation rows of
// one expert in shared memory.
constexpr int kTcW = 128;        // weight rows per work item (MMA M)
constexpr int kTcK = 64;         // K per pipeline step (one 128-byte swizzle row of bf16)
constexpr int kTcRowsUp = 192;   // sorted rows per gate_up work item (MMA N, at most)
constexpr int kTcRowsDown = 128; // sorted rows per down work item (MMA N, at most)

// Expert weight formats: MXFP4 (E2M1 + E8M0 per 32), int4_per_group_32 with
// float32 group scales, or with bfloat16 group scales.
enum class WeightKind : int { kMxfp4 = 0, kInt4 = 1, kInt4Bf16 = 2 };

// Bytes of one 32-group scale.
__host__ __device__ constexpr int scale_bytes(WeightKind k) { return k == WeightKind::kMxfp4 ? 1 : k == WeightKind::kInt4 ? 4 : 2; }

// Optional inputs of a call (moe_options_t), as the kernels read them.
struct LayerOptions {
  const uint16_t* b13 = nullptr;   // bf16 [E][2I], added to the gate_up outputs
  const uint16_t* b2 = nullptr;    // bf16 [E][H], added to each expert's output
  const int32_t* emap = nullptr;   // [G] global expert id -> local id or -1
  int G = 0;
  int rwi = 0;                     // router weight on the input, unweighted combine
  int aq = 0;                      // activation quantisation of both GEMM inputs (ActQuant)
  float s13 = 1.f, s2 = 1.f;       // static FP8 input scales of the gate_up / down GEMMs
  float clamp = 0.f;               // swiglu_limit: gate_up outputs clamped to [-clamp, clamp]; 0 = off
};

// Byte offsets of the workspace regions for one problem.
// Words between the CTAs of the fused decode kernel: an epoch (word 0) and
// one publication flag per CTA from word kSyncFlagsOffset on.
constexpr int kSyncFlagsOffset = 32;
constexpr int kMaxSyncCtas = 1024;
constexpr int kSyncWords = kSyncFlagsOffset + kMaxSyncCtas;
// Every workspace starts with the status word (a 256-byte region) and then
// the synchronisation words, whatever the problem.
constexpr size_t kStatusOffset = 0;
constexpr size_t kSyncOffset = 256;

struct Workspace {
  size_t status, sync, counts, offsets, active, n_active, gprefix, sorted_pair, pair_pos, mtiles, n_mtiles, mtiles_dn,
      n_mtiles_dn, rhist, rrank;
  size_t abuf, ybuf;        // decode: f32 [P][I], f32 [P][H]
  size_t xs, af, a16, aexp, outacc;  // prefill: bf16 [P][H], f32 [P][I], f16 [P][I], i32 [P], f32 [T][H]
  size_t total;
  bool prefill;
};

bool dims_valid(const moe_dims_t* d);
bool use_prefill(const moe_dims_t* d, WeightKind kind);
Workspace workspace_layout(const moe_dims_t* d, WeightKind kind);

// Device view of the routing result inside a workspace.
struct RouteOut {
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  int32_t* active;       // [E] ids of experts with >= 1 pair, ascending
  int32_t* n_active;     // [1]
  int32_t* gprefix;      // [E+1] exclusive prefix over active experts of ceil(count / kMoeGroup)
  int32_t* sorted_pair;  // [P]
  int32_t* pair_pos;     // [P]
  // tensor-core path: (expert << 20 | tile index) per row tile of an expert,
  // tiles of kTcRowsUp rows for gate_up and of kTcRowsDown rows for down
  int32_t* mtiles;       // [P / kTcRowsUp + E + 1]
  int32_t* n_mtiles;     // [1]
  int32_t* mtiles_dn;    // [P / kTcRowsDown + E + 1]
  int32_t* n_mtiles_dn;  // [1]
  uint32_t* status = nullptr;  // the call's status word (checked build), or none
};

// Launch ``kern`` on ``s``; with ``pdl`` the launch may begin before the previous
// kernel on the stream finishes (the kernel must call grid_dep_wait() before
// reading that kernel's results); with ``cooperative`` every CTA of the grid is
// resident at once, or the launch fails (for kernels whose CTAs wait on one
// another).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          bool cooperative, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Bounded-wait settings of one call: the limit of every wait in its kernels
// and, for tests of the give-up path only, extra CTAs the fused decode
// kernel's cross-CTA wait expects beyond its grid (so that wait runs out).
struct WaitSettings {
  uint64_t limit_ns = kWaitLimitNs;
  int extra_waiters = 0;
};
// Settings for the next call made from this host thread (moe_set_wait_limit);
// taking them resets the hook to the defaults.
WaitSettings take_wait_settings();

// Copy the status word of workspace ``ws`` to *status, then clear it and the
// synchronisation words (synchronises ``s``).
int read_and_clear_status(uint8_t* ws, uint32_t* status, cudaStream_t s);

// Benchmark timing hook (moe_set_timing_events): record the caller's event
// before (end = false) or after (end = true) kernel ``index`` of this call.
void timing_mark(int index, bool end, cudaStream_t s);

// Pairs above which (up to kRouteTwoPassMax) the grouping runs as two kernels
// over chunks of 1024 pairs (per-chunk counts and ranks, then placement);
// ``hist`` [ceil(P / 1024)][E] and ``rank`` [P] are their scratch (null: one
// CTA sorts everything).
constexpr long long kRouteTwoPassMax = 1ll << 20;
bool route_two_pass(long long P);
cudaError_t launch_route(const int32_t* topk_ids, int E, int T, int topk, const int32_t* emap, int G,
                         const RouteOut& r, int make_mtiles, cudaStream_t s, int32_t* hist = nullptr,
                         int32_t* rank = nullptr);

cudaError_t launch_router_topk(const float* logits, int T, int G, int topk, int renorm, int32_t* ids, float* w,
                               cudaStream_t s);

// out_s: float32 scales, or bf16 (uint16) with ``bf16``.
cudaError_t launch_requant(const uint8_t* w, const uint8_t* scale, uint8_t* out_q, void* out_s,
                           long long n_groups, bool bf16, cudaStream_t s);

struct DecodeArgs {
  WeightKind kind;
  int E, H, I, topk, T;
  const void* x;          // bf16 [T][H]
  const float* topk_w;    // [T][topk]
  const int32_t* topk_ids;
  const uint8_t* w13;     // packed [E][2I][H/2]
  const void* w13_s;      // u8 or f32 [E][2I][H/32]
  const uint8_t* w2;      // packed [E][H][I/2]
  const void* w2_s;       // u8 or f32 [E][H][I/32]
  void* out;              // bf16 [T][H]
  RouteOut route;
  float* abuf;            // [P][I], rows by sorted position
  float* ybuf;            // [P][H], rows by flat pair index
  uint32_t* status;
  uint32_t* sync;         // [kSyncWords] epoch and per-CTA flags of the fused kernel
  int num_sms;
  WaitSettings wait;
  LayerOptions opt;
};

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// Activation quantiser (ActQuant aq = 1 MXFP4 or 2 FP8) of rows x K values
// (bf16, or f32 with src_f32): codes to q, MX scale bytes to qs.
cudaError_t launch_act_quant(int aq, const void* x, bool src_f32, long long rows, int K, float s, uint8_t* q,
                             uint8_t* qs, int num_sms, cudaStream_t st);

struct PrefillArgs {
  int E, H, I, topk, T;
  const void* x;
  const float* topk_w;
  const int32_t* topk_ids;
  WeightKind kind;
  const uint8_t* w13;
  const void* w13_s;  // E8M0 bytes (MXFP4) or fp32 (int4) [E][2I][H/32]
  const uint8_t* w2;
  const void* w2_s;   // [E][H][I/32]
  void* out;
  RouteOut route;
  void* xs;       // bf16 [P][H]
  float* af;      // f32 [P][I]: the activated intermediate
  void* a16;      // f16 [P][I]: the same, row i scaled by 2^aexp[i]
  int32_t* aexp;  // [P]
  float* outacc;  // f32 [T][H]
  uint32_t* status;
  int num_sms;
  uint64_t wait_ns;
  LayerOptions opt;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);

}  // namespace moe
