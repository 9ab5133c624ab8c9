// Allocation-free variant of the MXFP4 MoE forward.
//
// moe_a16w4_mxfp4 needs a caller-provided workspace.  Some callers cannot
// allocate device memory at the point where they run the layer: code that
// must not call cudaMalloc (or a framework allocator) on its serving thread,
// plugins handed only input and output pointers by a host program that owns
// all allocation, or embedders whose memory is fully reserved up front.  For
// them this file keeps one fixed scratch array in device memory, sized for
// the weight-streaming (decode) kernels at small batches, and runs the same
// kernels on it.
#include <mutex>

#include "moe_internal.h"

namespace moe {

namespace {

// Largest workspace the variant can serve: 16 MiB covers the 112-expert,
// H = 3584, I = 3072, top-15 layer up to 32 tokens (about 12.8 MB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// One copy per GPU that loads the library, held until the process exits.
// Host code must not use this name as a device address; the address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

}  // namespace moe

extern "C" int moe_a16w4_mxfp4_noalloc(const moe_dims_t* d, const void* x, const int32_t* topk_ids,
                                       const float* topk_w, const uint8_t* w13, const uint8_t* w13_scale,
                                       const uint8_t* w2, const uint8_t* w2_scale, void* out, void* stream) {
  if (!d) return MOE_ERR_NULL;
  if (d->path == MOE_PATH_PREFILL) return MOE_ERR_BAD_DIMS;
  moe_dims_t dd = *d;
  dd.path = MOE_PATH_DECODE;
  if (!moe::dims_valid(&dd)) return MOE_ERR_BAD_DIMS;
  const size_t need = moe_workspace_bytes(&dd);
  if (need > moe::kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  if (dd.T == 0) return moe_a16w4_mxfp4(&dd, x, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, out, nullptr, 0,
                                        stream);
  void* scratch = nullptr;
  const int rc = moe::scratch_for_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_a16w4_mxfp4(&dd, x, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, out, scratch,
                         moe::kNoAllocScratchBytes, stream);
}

extern "C" int moe_noalloc_read_status(uint32_t* status, void* stream) {
  if (!status) return MOE_ERR_NULL;
  void* scratch = nullptr;
  const int rc = moe::scratch_for_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  return moe::read_and_clear_status(reinterpret_cast<uint8_t*>(scratch), status,
                                    reinterpret_cast<cudaStream_t>(stream));
}
