// C ABI entry points: argument checks, workspace layout, kernel sequencing.
#include <stdio.h>

#include "moe_internal.h"

namespace moe {

namespace {

struct TimingHook {
  cudaEvent_t ev[16];
  int n = 0;
};
thread_local TimingHook g_timing;
thread_local WaitSettings g_wait;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The library is built for sm_103a only.
int check_device(int* num_sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
  if (num_sms && cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

RouteOut route_view(uint8_t* ws, const Workspace& L) {
  RouteOut r;
  r.counts = reinterpret_cast<int32_t*>(ws + L.counts);
  r.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  r.active = reinterpret_cast<int32_t*>(ws + L.active);
  r.n_active = reinterpret_cast<int32_t*>(ws + L.n_active);
  r.gprefix = reinterpret_cast<int32_t*>(ws + L.gprefix);
  r.sorted_pair = reinterpret_cast<int32_t*>(ws + L.sorted_pair);
  r.pair_pos = reinterpret_cast<int32_t*>(ws + L.pair_pos);
  r.mtiles = reinterpret_cast<int32_t*>(ws + L.mtiles);
  r.n_mtiles = reinterpret_cast<int32_t*>(ws + L.n_mtiles);
  r.mtiles_dn = reinterpret_cast<int32_t*>(ws + L.mtiles_dn);
  r.n_mtiles_dn = reinterpret_cast<int32_t*>(ws + L.n_mtiles_dn);
  r.status = reinterpret_cast<uint32_t*>(ws + L.status);
  return r;
}

int common_checks(const moe_dims_t* d, const void* x, const int32_t* ids, const float* tw, const void* w13,
                  const void* s13, const void* w2, const void* s2, void* out, void* ws, size_t ws_bytes,
                  WeightKind kind) {
  if (!d) return MOE_ERR_NULL;
  if (d->act != MOE_ACT_SWIGLU) return MOE_ERR_UNSUPPORTED_ACT;
  if (!dims_valid(d)) return MOE_ERR_BAD_DIMS;
  if (d->path == MOE_PATH_PREFILL && !use_prefill(d, kind)) return MOE_ERR_BAD_DIMS;
  if (d->T == 0) return MOE_OK;
  if (!x || !ids || !tw || !w13 || !s13 || !w2 || !s2 || !out || !ws) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(s13, 16) || !aligned(w2, 16) || !aligned(s2, 16) ||
      !aligned(out, 16) || !aligned(ws, 256) || !aligned(ids, 4) || !aligned(tw, 4))
    return MOE_ERR_ALIGN;
  if (ws_bytes < workspace_layout(d, kind).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Options of a call from the public struct (NULL = none), checked.
int read_options(const moe_options_t* o, LayerOptions* lo) {
  *lo = LayerOptions{};
  if (!o) return MOE_OK;
  if (o->router_weight_on_input != 0 && o->router_weight_on_input != 1) return MOE_ERR_BAD_DIMS;
  if (o->expert_map && (o->global_num_experts < 1 || o->global_num_experts > (1 << 20))) return MOE_ERR_BAD_DIMS;
  if (!aligned(o->w13_bias, 2) || !aligned(o->w2_bias, 2) || !aligned(o->expert_map, 4)) return MOE_ERR_ALIGN;
  lo->b13 = reinterpret_cast<const uint16_t*>(o->w13_bias);
  lo->b2 = reinterpret_cast<const uint16_t*>(o->w2_bias);
  lo->emap = o->expert_map;
  lo->G = o->expert_map ? o->global_num_experts : 0;
  lo->rwi = o->router_weight_on_input;
  if (o->act_quant < MOE_AQ_NONE || o->act_quant > MOE_AQ_FP8) return MOE_ERR_BAD_DIMS;
  lo->aq = o->act_quant;
  if (lo->aq == MOE_AQ_FP8) {
    // static scales: finite and positive (the comparisons are false for NaN)
    if (!(o->w13_input_scale > 0.f && o->w13_input_scale <= 3.0e38f)) return MOE_ERR_BAD_DIMS;
    if (!(o->w2_input_scale > 0.f && o->w2_input_scale <= 3.0e38f)) return MOE_ERR_BAD_DIMS;
    lo->s13 = o->w13_input_scale;
    lo->s2 = o->w2_input_scale;
  }
  if (!(o->swiglu_limit >= 0.f && o->swiglu_limit <= 3.0e38f)) return MOE_ERR_BAD_DIMS;  // NaN fails too
  lo->clamp = o->swiglu_limit;
  // the schemes quantise the activations of MXFP4-weight layers; the router
  // weight on the input is not modelled together with them
  if (lo->aq != MOE_AQ_NONE && lo->rwi) return MOE_ERR_BAD_DIMS;
  return MOE_OK;
}

int run_moe(const moe_dims_t* d, const void* x, const int32_t* ids, const float* tw, const uint8_t* w13,
            const void* s13, const uint8_t* w2, const void* s2, const moe_options_t* options, void* out,
            void* workspace, size_t ws_bytes, void* stream, WeightKind kind) {
  const WaitSettings wait = take_wait_settings();  // the hook applies to this call only
  int rc = common_checks(d, x, ids, tw, w13, s13, w2, s2, out, workspace, ws_bytes, kind);
  if (rc != MOE_OK) return rc;
  LayerOptions opt;
  rc = read_options(options, &opt);
  if (rc == MOE_OK && opt.aq != MOE_AQ_NONE && kind != WeightKind::kMxfp4) rc = MOE_ERR_BAD_DIMS;
  if (rc != MOE_OK || d->T == 0) return rc;
  int sms = 0;
  rc = check_device(&sms);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Workspace L = workspace_layout(d, kind);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const RouteOut r = route_view(ws, L);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);

  // small decode batches are grouped inside the decode kernels
  const bool route_kernel = L.prefill || (long long)d->T * d->topk > kMaxLocalRoutePairs;
  timing_mark(0, false, s);
  if (route_kernel && launch_route(ids, d->E, d->T, d->topk, opt.emap, opt.G, r, L.prefill ? 1 : 0, s,
                                   reinterpret_cast<int32_t*>(ws + L.rhist),
                                   reinterpret_cast<int32_t*>(ws + L.rrank)) != cudaSuccess)
    return MOE_ERR_CUDA;
  timing_mark(0, true, s);
  cudaError_t e;
  if (L.prefill) {
    PrefillArgs a{};
    a.E = d->E; a.H = d->H; a.I = d->I; a.topk = d->topk; a.T = d->T;
    a.x = x; a.topk_w = tw; a.topk_ids = ids;
    a.kind = kind;
    a.w13 = w13; a.w13_s = s13;
    a.w2 = w2; a.w2_s = s2;
    a.out = out; a.route = r;
    a.xs = ws + L.xs;
    a.af = reinterpret_cast<float*>(ws + L.af);
    a.a16 = ws + L.a16;
    a.aexp = reinterpret_cast<int32_t*>(ws + L.aexp);
    a.outacc = reinterpret_cast<float*>(ws + L.outacc);
    a.status = status; a.num_sms = sms;
    a.wait_ns = wait.limit_ns;
    a.opt = opt;
    e = launch_prefill(a, s);
  } else {
    DecodeArgs a{};
    a.kind = kind;
    a.E = d->E; a.H = d->H; a.I = d->I; a.topk = d->topk; a.T = d->T;
    a.x = x; a.topk_w = tw; a.topk_ids = ids;
    a.w13 = w13; a.w13_s = s13; a.w2 = w2; a.w2_s = s2;
    a.out = out; a.route = r;
    a.abuf = reinterpret_cast<float*>(ws + L.abuf);
    a.ybuf = reinterpret_cast<float*>(ws + L.ybuf);
    a.status = status; a.num_sms = sms;
    a.sync = reinterpret_cast<uint32_t*>(ws + L.sync);
    a.wait = wait;
    a.opt = opt;
    e = launch_decode(a, s);
  }
  g_timing.n = 0;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int read_and_clear_status(uint8_t* ws, uint32_t* status, cudaStream_t s) {
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws + kStatusOffset, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  // the status word, and the fused decode kernel's epoch and flags (a kernel
  // that gave up a wait may have left them inconsistent)
  if (cudaMemsetAsync(ws + kStatusOffset, 0, sizeof(v), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws + kSyncOffset, 0, 4 * kSyncWords, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

WaitSettings take_wait_settings() {
  const WaitSettings w = g_wait;
  g_wait = WaitSettings{};
  return w;
}

void timing_mark(int index, bool end, cudaStream_t s) {
  if (index >= g_timing.n) return;
  cudaEvent_t ev = g_timing.ev[2 * index + (end ? 1 : 0)];
  // Under stream capture only an external record becomes an event node of the
  // graph; outside capture a plain record is used.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

bool dims_valid(const moe_dims_t* d) {
  if (!d) return false;
  if (d->E < 1 || d->E > kMaxExperts) return false;
  // the weight-streaming kernels stage 32 weight rows of the whole K per
  // pipeline slot and need two slots in shared memory: K <= 4096
  if (d->H < 64 || d->H > 4096 || d->H % 64) return false;
  if (d->I < 64 || d->I > 4096 || d->I % 64) return false;
  if (d->topk < 1 || d->topk > 64) return false;
  if (d->T < 0 || (long long)d->T * d->topk > (1ll << 24)) return false;
  if (d->path < MOE_PATH_AUTO || d->path > MOE_PATH_PREFILL) return false;
  return true;
}

bool use_prefill(const moe_dims_t* d, WeightKind kind) {
  (void)kind;  // both weight formats have tensor-core kernels
  // the tensor-core kernels load packed weights and scales in 256-of-K groups
  // and their gather kernel handles rows of at most 4096 elements
  const bool ok = (d->H % 512 == 0) && (d->I % 512 == 0) && d->H <= 4096 && d->I <= 4096 && kPrefillAvailable;
  if (d->path == MOE_PATH_PREFILL) return ok;
  if (d->path == MOE_PATH_DECODE) return false;
  return ok && d->T >= kPrefillMinTokens;
}

Workspace workspace_layout(const moe_dims_t* d, WeightKind kind) {
  Workspace L{};
  const size_t E = d->E, P = (size_t)d->T * d->topk, H = d->H, I = d->I, T = d->T;
  L.prefill = use_prefill(d, kind);
  size_t o = 0;
  L.status = o; o = align256(o + 256);
  L.sync = o; o = align256(o + 4 * kSyncWords);
  static_assert(kStatusOffset == 0 && kSyncOffset == 256, "status and sync words lead every workspace");
  L.counts = o; o = align256(o + 4 * E);
  L.offsets = o; o = align256(o + 4 * (E + 1));
  L.active = o; o = align256(o + 4 * E);
  L.n_active = o; o = align256(o + 4);
  L.gprefix = o; o = align256(o + 4 * (E + 1));
  L.sorted_pair = o; o = align256(o + 4 * P);
  L.pair_pos = o; o = align256(o + 4 * P);
  L.mtiles = o; o = align256(o + 4 * (P / kTcRowsUp + E + 1));
  L.n_mtiles = o; o = align256(o + 4);
  L.mtiles_dn = o; o = align256(o + 4 * (P / kTcRowsDown + E + 1));
  L.n_mtiles_dn = o; o = align256(o + 4);
  // scratch of the two-kernel grouping of large batches
  L.rhist = o; o = align256(o + (route_two_pass((long long)P) ? 4 * ((P + 1023) / 1024) * E : 0));
  L.rrank = o; o = align256(o + (route_two_pass((long long)P) ? 4 * P : 0));
  if (L.prefill) {
    L.xs = o; o = align256(o + 2 * P * H);
    L.af = o; o = align256(o + 4 * P * I);
    L.a16 = o; o = align256(o + 2 * P * I);
    L.aexp = o; o = align256(o + 4 * P);
    L.outacc = o; o = align256(o + 4 * T * H);
  } else {
    L.abuf = o; o = align256(o + 4 * P * I);
    L.ybuf = o; o = align256(o + 4 * P * H);
  }
  L.total = o;
  return L;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_dims_t* d) {
  if (!dims_valid(d)) return 0;
  return workspace_layout(d, WeightKind::kMxfp4).total > workspace_layout(d, WeightKind::kInt4).total
             ? workspace_layout(d, WeightKind::kMxfp4).total
             : workspace_layout(d, WeightKind::kInt4).total;
}

int moe_a16w4_mxfp4(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                    const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2, const uint8_t* w2_scale,
                    void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return run_moe(d, x, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, nullptr, out, workspace, workspace_bytes,
                 stream, WeightKind::kMxfp4);
}

int moe_a16w4_int4g32(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                      const uint8_t* w13_q, const float* w13_s, const uint8_t* w2_q, const float* w2_s, void* out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return run_moe(d, x, topk_ids, topk_w, w13_q, w13_s, w2_q, w2_s, nullptr, out, workspace, workspace_bytes,
                 stream, WeightKind::kInt4);
}

int moe_a16w4_mxfp4_ex(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                       const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2, const uint8_t* w2_scale,
                       const moe_options_t* opt, void* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return run_moe(d, x, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, opt, out, workspace, workspace_bytes,
                 stream, WeightKind::kMxfp4);
}

int moe_a16w4_int4g32_ex(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                         const uint8_t* w13_q, const float* w13_s, const uint8_t* w2_q, const float* w2_s,
                         const moe_options_t* opt, void* out, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return run_moe(d, x, topk_ids, topk_w, w13_q, w13_s, w2_q, w2_s, opt, out, workspace, workspace_bytes, stream,
                 WeightKind::kInt4);
}

int moe_a16w4_int4g32_bf16s(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13_q, const void* w13_s, const uint8_t* w2_q, const void* w2_s,
                            void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return run_moe(d, x, topk_ids, topk_w, w13_q, w13_s, w2_q, w2_s, nullptr, out, workspace, workspace_bytes,
                 stream, WeightKind::kInt4Bf16);
}

int moe_a16w4_int4g32_bf16s_ex(const moe_dims_t* d, const void* x, const int32_t* topk_ids, const float* topk_w,
                               const uint8_t* w13_q, const void* w13_s, const uint8_t* w2_q, const void* w2_s,
                               const moe_options_t* opt, void* out, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return run_moe(d, x, topk_ids, topk_w, w13_q, w13_s, w2_q, w2_s, opt, out, workspace, workspace_bytes, stream,
                 WeightKind::kInt4Bf16);
}

static int requant_entry(int32_t E, int32_t N, int32_t K, const uint8_t* w, const uint8_t* scale, uint8_t* out_q,
                         void* out_s, int32_t experts_per_chunk, bool bf16, void* stream) {
  if (E < 1 || N < 1 || K < 32 || K % 32 || experts_per_chunk < 1) return MOE_ERR_BAD_DIMS;
  if (!w || !scale || !out_q || !out_s) return MOE_ERR_NULL;
  if (!aligned(w, 16) || !aligned(out_q, 16) || !aligned(out_s, 16)) return MOE_ERR_ALIGN;
  const int rc = check_device(nullptr);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long groups_per_expert = (long long)N * (K / 32);
  for (int lo = 0; lo < E; lo += experts_per_chunk) {
    const int hi = lo + experts_per_chunk < E ? lo + experts_per_chunk : E;
    const long long g0 = (long long)lo * groups_per_expert;
    void* os = reinterpret_cast<uint8_t*>(out_s) + g0 * (bf16 ? 2 : 4);
    if (launch_requant(w + g0 * 16, scale + g0, out_q + g0 * 16, os, (long long)(hi - lo) * groups_per_expert, bf16,
                       s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int requant_mxfp4_to_int4g32(int32_t E, int32_t N, int32_t K, const uint8_t* w, const uint8_t* scale,
                             uint8_t* out_q, float* out_s, int32_t experts_per_chunk, void* stream) {
  return requant_entry(E, N, K, w, scale, out_q, out_s, experts_per_chunk, false, stream);
}

int requant_mxfp4_to_int4g32_bf16s(int32_t E, int32_t N, int32_t K, const uint8_t* w, const uint8_t* scale,
                                   uint8_t* out_q, void* out_s, int32_t experts_per_chunk, void* stream) {
  return requant_entry(E, N, K, w, scale, out_q, out_s, experts_per_chunk, true, stream);
}

int moe_route(const moe_dims_t* d, const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
              int32_t* sorted_pair, int32_t* pair_pos, void* stream) {
  if (!d) return MOE_ERR_NULL;
  if (d->E < 1 || d->E > kMaxExperts || d->topk < 1 || d->topk > 64 || d->T < 0 ||
      (long long)d->T * d->topk > (1ll << 24))
    return MOE_ERR_BAD_DIMS;
  if (!counts || !offsets) return MOE_ERR_NULL;
  if (d->T > 0 && (!topk_ids || !sorted_pair || !pair_pos)) return MOE_ERR_NULL;
  const int rc = check_device(nullptr);
  if (rc != MOE_OK) return rc;
  // Only the four grouping outputs are requested; the kernel skips the
  // auxiliary lists when their pointers are null.
  RouteOut r{};
  r.counts = counts;
  r.offsets = offsets;
  r.sorted_pair = sorted_pair;
  r.pair_pos = pair_pos;
  if (launch_route(topk_ids, d->E, d->T, d->topk, nullptr, 0, r, 0, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_router_topk(const float* logits, int32_t T, int32_t G, int32_t topk, int32_t renormalize,
                    int32_t* topk_ids, float* topk_w, void* stream) {
  if (T < 0 || G < 1 || G > 1024 || topk < 1 || topk > 64 || topk > G || (renormalize != 0 && renormalize != 1) ||
      (long long)T * G > (1ll << 31) - 1)
    return MOE_ERR_BAD_DIMS;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_NULL;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_ERR_ALIGN;
  const int rc = check_device(nullptr);
  if (rc != MOE_OK) return rc;
  return launch_router_topk(logits, T, G, topk, renormalize, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_quantize_act(int32_t act_quant, const void* x, int32_t x_is_f32, int64_t rows, int32_t K, float scale,
                     uint8_t* q, uint8_t* q_scale, void* stream) {
  if (act_quant != MOE_AQ_MXFP4 && act_quant != MOE_AQ_FP8) return MOE_ERR_BAD_DIMS;
  if ((x_is_f32 != 0 && x_is_f32 != 1) || rows < 0 || rows > (1ll << 31) || K < 32 || K % 32 || K > (1 << 20))
    return MOE_ERR_BAD_DIMS;
  if (act_quant == MOE_AQ_FP8 && !(scale > 0.f && scale <= 3.0e38f)) return MOE_ERR_BAD_DIMS;
  if (rows == 0) return MOE_OK;
  if (!x || !q || (act_quant == MOE_AQ_MXFP4 && !q_scale)) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(q, 16)) return MOE_ERR_ALIGN;
  int sms = 0;
  const int rc = check_device(&sms);
  if (rc != MOE_OK) return rc;
  return launch_act_quant(act_quant, x, x_is_f32 == 1, rows, K, scale, q, q_scale, sms,
                          reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_read_status(const moe_dims_t* d, void* workspace, uint32_t* status, void* stream) {
  if (!d || !workspace || !status) return MOE_ERR_NULL;
  if (!dims_valid(d)) return MOE_ERR_BAD_DIMS;
  return read_and_clear_status(reinterpret_cast<uint8_t*>(workspace), status, reinterpret_cast<cudaStream_t>(stream));
}

int moe_set_timing_events(void* const* events, int32_t n) {
  if (n < 0 || n > 8) return MOE_ERR_BAD_DIMS;
  if (n > 0 && !events) return MOE_ERR_NULL;
  for (int i = 0; i < 2 * n; ++i) g_timing.ev[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  g_timing.n = n;
  return MOE_OK;
}

int moe_set_wait_limit(uint64_t limit_ns, int32_t extra_waiters) {
  if (limit_ns == 0 || extra_waiters < 0 || extra_waiters > 64) return MOE_ERR_BAD_DIMS;
  g_wait.limit_ns = limit_ns;
  g_wait.extra_waiters = extra_waiters;
  return MOE_OK;
}

const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_BAD_DIMS: return "unsupported problem size";
    case MOE_ERR_ALIGN: return "pointer not aligned as documented";
    case MOE_ERR_UNSUPPORTED_ACT: return "unsupported activation (only SwiGLU is implemented)";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE: return "device is not a compute capability 10.3 GPU";
    default: return "unknown error";
  }
}

int moe_abi_version(void) { return 104; }

}  // extern "C"
