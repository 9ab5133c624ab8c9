// MXFP4 -> int4_per_group_32 requantisation (load time, lossy, opt-in).
//
// Follows Mxfp4MoEMethod._setup_kernel_k3_situ_gfx942 (vLLM quantization/mxfp4
// API page): decode E2M1 elements and the E8M0 block scale, multiply, cast to
// bf16 (exact for these values), then symmetric int4 per 32-group with
//   scale = fl32(amax / 7),  q = round_half_even(fl32(w / scale)), q in [-8, 7],
// an all-zero group giving scale 0 and q 0.
//
// One thread per 32-group and iteration (four per thread in flight): 16 bytes
// in, one scale byte in, 16 bytes and one float out, all coalesced; one wave
// of resident CTAs.  HBM-bound.  Division-free fast path: inside the
// normal float32 range every element is c * 2^(s-127) and the group maximum is
// cmax * 2^(s-127), so fl32(w / fl32(amax / 7)) equals
// fl32(c / fl32(cmax / 7)) -- the power of two cancels exactly.  The quotient
// therefore depends only on the two codes: tables built at kernel start with
// the same IEEE round-to-nearest divisions give, per cmax, the output byte of
// every packed input byte (two signed codes), so a group costs sixteen
// shared-memory byte loads, each addressed by one byte permute, instead of
// 32 divisions; likewise fl32(amax / 7) = fl32(cmax / 7) * 2^(s-127).  The
// largest code itself comes from byte permutes (one-hot bytes, then the
// highest set bit of their OR), which keeps the integer work per group below
// the HBM time.  Groups whose scale byte puts values near the subnormal range
// or near overflow take the per-element division path, so results are
// bit-exact for every scale byte in [0, 252].
//
// bf16 scales (the "groupwise bf16 scales" of the PR #51274 commit message):
// the scale is rounded to bf16 (nearest even) before the elements are divided
// by it; bf16 rounding commutes with the power of two like float32 rounding
// does, so the same two-code tables hold, built from the rounded scales.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kRequantThreads = 256;
constexpr int kGroupsPerIter = 4;  // 32-groups per thread and loop iteration
// Scale bytes inside which the table path is exact (values, amax/7 and the
// quotients are normal float32 numbers and nothing overflows).
constexpr uint32_t kFastLo = 8, kFastHi = 250;

// Magnitude of an E2M1 code (low 3 bits): exponent field e = c>>1 (bias 1),
// mantissa bit c&1; e = 0 is the subnormal 0.5 * mantissa.
__device__ __forceinline__ float e2m1_mag(uint32_t c) {
  c &= 7u;
  const uint32_t normal = (((c >> 1) + 126u) << 23) | ((c & 1u) << 22);
  return __uint_as_float(c >= 2u ? normal : (c ? 0x3F000000u : 0u));
}

// One packed word (four bytes, eight E2M1 codes) -> its four output bytes
// (eight int4 codes) through the byte table of the group's largest code:
// row_sel = cmax << 8, so one byte permute forms each entry's index
// cmax * 256 + byte into the [8][256] table.
__device__ __forceinline__ uint32_t lookup_word(uint32_t w, uint32_t row_sel, const uint8_t* tab) {
  const uint32_t b0 = tab[prmt(w, row_sel, 0x7650u)], b1 = tab[prmt(w, row_sel, 0x7651u)];
  const uint32_t b2 = tab[prmt(w, row_sel, 0x7652u)], b3 = tab[prmt(w, row_sel, 0x7653u)];
  return prmt(prmt(b0, b1, 0x0040u), prmt(b2, b3, 0x0040u), 0x5410u);
}

// One group: 16 packed bytes v and scale byte s -> 16 bytes of int4 codes and
// the fp32 scale.  ltab[cmax][byte]: the output byte of a packed byte (two
// signed codes) in a group whose largest magnitude code is cmax; lut_s[cmax]
// = fl32(cmax / 7).
template <bool BF16>
__device__ __forceinline__ void requant_group(const uint4& v, uint32_t s, const uint8_t (*ltab)[256],
                                              const float* lut_s, uint4& q_out, float& s_out) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  // largest magnitude code in the group: a byte permute turns four
  // magnitudes (selector nibbles, sign bits cleared) into one-hot bytes
  // 1 << m, the OR of all of them has bit cmax as its highest
  uint32_t oh = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t mg = wd[i] & 0x77777777u;
    oh |= prmt(0x08040201u, 0x80402010u, mg) | prmt(0x08040201u, 0x80402010u, mg >> 16);
  }
  oh |= oh >> 16;
  oh |= oh >> 8;
  const uint32_t cmax = 31u - __clz((oh & 0xFFu) | 1u);
  const float sc_unit = e8m0_to_float(s);
  uint32_t oq[4];
  float oscale;
  if (cmax == 0) {
    oq[0] = oq[1] = oq[2] = oq[3] = 0u;
    oscale = 0.f;
  } else if (s >= kFastLo && s <= kFastHi) {
    // fl32(cmax * 2^(s-127) / 7) = fl32(cmax / 7) * 2^(s-127): the product is a
    // normal float for these scale bytes, so the power of two commutes with
    // the rounding
    oscale = lut_s[cmax] * sc_unit;
#pragma unroll
    for (int i = 0; i < 4; ++i) oq[i] = lookup_word(wd[i], cmax << 8, &ltab[0][0]);
  } else {
    // exact per-element path (values near the subnormal range or near overflow)
    const float amax = e2m1_mag(cmax) * sc_unit;
    oscale = __fdiv_rn(amax, 7.0f);
    if (BF16) oscale = bf16_lo(f32_to_bf16_bits(oscale));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t r = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t c = (wd[i] >> (4 * j)) & 0xFu;
        float val = e2m1_mag(c) * sc_unit;
        val = (c & 8u) ? -val : val;
        int q = oscale > 0.f ? __float2int_rn(__fdiv_rn(val, oscale)) : 0;
        q = min(max(q, -8), 7);
        r |= uint32_t(q & 0xF) << (4 * j);
      }
      oq[i] = r;
    }
  }
  q_out = make_uint4(oq[0], oq[1], oq[2], oq[3]);
  s_out = oscale;
}

// BF16: scales rounded to bf16 before the division, stored as bf16 (out_s
// holds uint16 then).
template <bool BF16>
__global__ void __launch_bounds__(kRequantThreads) requant_kernel(const uint8_t* __restrict__ w,
                                                                  const uint8_t* __restrict__ scale,
                                                                  uint8_t* __restrict__ out_q,
                                                                  void* __restrict__ out_s, int n_groups) {
  // per cmax (largest magnitude code of a group, 1..7): fl32(cmax / 7), the
  // int4 code of each signed E2M1 code, and from those the output byte of
  // every packed byte (two codes)
  __shared__ float lut_s[8];
  __shared__ uint8_t qcode[8][16];
  __shared__ uint8_t ltab[8][256];
  if (threadIdx.x < 8) {
    float u = threadIdx.x ? __fdiv_rn(e2m1_mag(threadIdx.x), 7.0f) : 0.f;
    if (BF16) u = bf16_lo(f32_to_bf16_bits(u));
    lut_s[threadIdx.x] = u;
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    const uint32_t cm = threadIdx.x >> 4, c = threadIdx.x & 15;
    int q = 0;
    if (cm > 0) {
      q = __float2int_rn(__fdiv_rn(e2m1_mag(c), lut_s[cm]));
      q = min(max(q, -8), 7);
      if (c & 8u) q = -q;
    }
    qcode[cm][c] = (uint8_t)(q & 0xF);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) {
    const int cm = i >> 8, b = i & 255;
    ltab[cm][b] = (uint8_t)(qcode[cm][b & 15] | (qcode[cm][b >> 4] << 4));
  }
  __syncthreads();

  // kGroupsPerIter groups per thread and iteration, all loads issued before
  // any arithmetic, so that many 16-byte loads per thread are in flight
  // 32-bit group indices (the host launches at most 2^30 groups at a time)
  const int stride = gridDim.x * blockDim.x;
  for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < n_groups; g += kGroupsPerIter * stride) {
    uint4 v[kGroupsPerIter];
    uint32_t sb[kGroupsPerIter];
#pragma unroll
    for (int i = 0; i < kGroupsPerIter; ++i) {
      const int gi = g + i * stride;
      v[i] = make_uint4(0, 0, 0, 0);
      sb[i] = 0;
      if (gi < n_groups) {
        v[i] = __ldcs(reinterpret_cast<const uint4*>(w) + gi);
        sb[i] = scale[gi];
      }
    }
#pragma unroll
    for (int i = 0; i < kGroupsPerIter; ++i) {
      const int gi = g + i * stride;
      if (gi < n_groups) {
        uint4 q;
        float o;
        requant_group<BF16>(v[i], sb[i], ltab, lut_s, q, o);
        __stcs(reinterpret_cast<uint4*>(out_q) + gi, q);
        // (o is a bf16 value here: its high half is exact)
        if (BF16) __stcs(reinterpret_cast<unsigned short*>(out_s) + gi, (unsigned short)(__float_as_uint(o) >> 16));
        else __stcs(reinterpret_cast<float*>(out_s) + gi, o);
      }
    }
  }
}

}  // namespace

cudaError_t launch_requant(const uint8_t* w, const uint8_t* scale, uint8_t* out_q, void* out_s,
                           long long n_groups, bool bf16, cudaStream_t s) {
  if (n_groups <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // one wave: as many CTAs as are resident at once (a second, partial wave
  // would leave most SMs idle at the end)
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, requant_kernel<false>, kRequantThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // pieces of at most 2^30 groups, so that the kernel indexes in 32 bits
  constexpr long long kPiece = 1ll << 30;
  for (long long g0 = 0; g0 < n_groups; g0 += kPiece) {
    const int n = (int)(n_groups - g0 < kPiece ? n_groups - g0 : kPiece);
    const long long want = (n + kRequantThreads - 1) / kRequantThreads;
    const long long resident = (long long)sms * per_sm;
    const int grid = (int)(want < resident ? want : resident);
    if (bf16)
      requant_kernel<true><<<grid, kRequantThreads, 0, s>>>(w + g0 * 16, scale + g0, out_q + g0 * 16,
                                                          reinterpret_cast<uint16_t*>(out_s) + g0, n);
    else
      requant_kernel<false><<<grid, kRequantThreads, 0, s>>>(w + g0 * 16, scale + g0, out_q + g0 * 16,
                                                           reinterpret_cast<float*>(out_s) + g0, n);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
