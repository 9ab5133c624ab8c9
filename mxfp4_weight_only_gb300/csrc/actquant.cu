// Activation quantiser of the W4A4 / W4A8 schemes (vLLM PR #39136:
// ``w_mxfp4_a_mxfp4``, ``w_mxfp4_a_fp8``) as a library call, built from the
// same device routines the layer kernels apply where they load a GEMM input.
// HBM-bound: one pass over the input, codes (and MX scales) written once.
#include "common.cuh"

namespace moe {

namespace {

// Thread i quantises the 8 values [8i, 8i + 8) of the flattened [rows][K]
// input (K % 32 == 0, so the 4 threads of a 32-block are lanes 4m .. 4m+3 of
// one warp).  The loop bound is uniform per block, so every lane of a warp
// reaches the block-maximum shuffles together.
template <bool SRC_F32>
__global__ void __launch_bounds__(256) act_quant_kernel(const void* __restrict__ x, long long n8, int aq, float s,
                                                        uint8_t* __restrict__ q, uint8_t* __restrict__ qs) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x; i0 < n8; i0 += stride) {
    const long long i = i0 + threadIdx.x;
    const bool valid = i < n8;
    float v[8];
    if (valid) {
      if (SRC_F32) {
        const float4* p = reinterpret_cast<const float4*>(x) + 2 * i;
        const float4 a = __ldcs(p), b = __ldcs(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      } else {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(x) + i);
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = 0.f;
    }
    if (aq == kActMxfp4) {
      uint32_t codes, sb;
      mx_quant8(v, codes, sb);
      if (valid) {
        reinterpret_cast<uint32_t*>(q)[i] = codes;
        if ((i & 3) == 0) qs[i >> 2] = (uint8_t)sb;
      }
    } else {
      uint32_t c0, c1;
      fp8_quant8(v, s, c0, c1);
      if (valid) reinterpret_cast<uint2*>(q)[i] = make_uint2(c0, c1);
    }
  }
}

}  // namespace

cudaError_t launch_act_quant(int aq, const void* x, bool src_f32, long long rows, int K, float s, uint8_t* q,
                             uint8_t* qs, int num_sms, cudaStream_t st) {
  const long long n8 = rows * (long long)(K / 8);
  if (n8 == 0) return cudaSuccess;
  const long long want = (n8 + 255) / 256;
  const int grid = (int)(want < (long long)num_sms * 8 ? want : (long long)num_sms * 8);
  if (src_f32) act_quant_kernel<true><<<grid, 256, 0, st>>>(x, n8, aq, s, q, qs);
  else act_quant_kernel<false><<<grid, 256, 0, st>>>(x, n8, aq, s, q, qs);
  return cudaGetLastError();
}

}  // namespace moe
