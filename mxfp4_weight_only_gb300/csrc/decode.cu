// Weight-streaming grouped GEMMs for small batches (decode), HBM-bound.
//
// The two stages of the fused MoE (Mxfp4MoEMethod.apply on the vLLM
// quantization/mxfp4 API page; gate_up ``w13`` then down ``w2``), for few
// tokens per expert:
//   gemm1:  h = W13[e] x  for every pair of expert e, fused SiLU-gated
//           activation a[j] = SiLU(h[j]) * h[I + j]  -> abuf (fp32, rows by
//           sorted pair position)
//   gemm2:  y = W2[e] a  -> ybuf (fp32, rows by flat pair index)
//   combine: out[t] = bf16( sum_k topk_w[t,k] * y[t*topk + k] ), k ascending.
//
// Work item = (active expert, 16 weight rows x all of K).  For gemm1 the 16
// rows are 8 gate rows j..j+7 and the matching 8 up rows I+j.., so the
// activation is local to the item.  Items are split into one contiguous run
// per CTA (one CTA per SM, persistent); consecutive items of one CTA share an
// expert, so its activations stay in registers across items.
//
// Per CTA: one producer warp streams each item's 16 weight rows (row-wise
// cp.async.bulk into a padded shared-memory stage, conflict-free for the
// consumers) and their scales through an mbarrier ring.  Fifteen consumer
// warps split K (16 warps per CTA: four per SM sub-partition); each turns its part of the packed rows into m16n8k16 f16 MMA
// operands (E2M1 pairs via cvt.rn.f16x2.e2m1x2, exact; int4 pairs via the
// 1024-offset f16 trick, exact), multiplies by up to 8 activation columns, and
// applies the per-32-block weight scale to each block's fp32 partial sum.
// Activations enter the MMA as f16 scaled by a power of two per (pair, warp
// K-range) so they cannot overflow; the scale is removed in fp32 afterwards.
// Partial sums of the consumer warps are reduced through shared memory.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kConsumerWarps = 15;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kRows = 16;          // weight rows per item
constexpr int kCols = 8;           // pairs per MMA column group
constexpr int kSmemBudget = 220 * 1024;

struct GemmParams {
  const uint8_t* w;        // packed weights [E][N][K/2]
  const void* ws;          // scales [E][N][K/32], u8 (E8M0) or f32
  int N, K, I;             // rows per expert, reduction size, I (gate/up split for gemm1)
  int tiles;               // items per expert
  const void* src;         // gemm1: x bf16 [T][K]; gemm2: abuf f32 [P][K]
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  const int32_t* sorted_pair;
  int topk;
  float* dst;              // gemm1: abuf [P][I]; gemm2: ybuf [P][N]
  uint32_t* status;
  int row_stride;          // bytes between staged weight rows (K/2 + 16)
  int srow_bytes;          // scale bytes per weight row
  int stage_bytes;
  int n_stages;
};

__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight packed int4 (two's complement) -> four f16x2, pairs (i, i+4).
__device__ __forceinline__ void int4x8_to_f16x8(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
  const uint32_t u = w ^ 0x88888888u;  // offset binary: q + 8
  const uint32_t magic = 0x64006400u;  // f16 1024 in both halves
  const uint32_t bias = 0x64086408u;   // f16 1032
  o0 = f16x2_sub((u & 0x000F000Fu) | magic, bias);
  o1 = f16x2_sub(((u >> 4) & 0x000F000Fu) | magic, bias);
  o2 = f16x2_sub(((u >> 8) & 0x000F000Fu) | magic, bias);
  o3 = f16x2_sub(((u >> 12) & 0x000F000Fu) | magic, bias);
}

template <bool GATE_UP>
__device__ __forceinline__ int item_row(int r, int j, int I) {
  if (GATE_UP) return r < 8 ? 8 * j + r : I + 8 * j + (r - 8);
  return kRows * j + r;
}

// Load 8 consecutive activation values of one row as float.
template <bool SRC_BF16>
__device__ __forceinline__ void load8(const void* row, int k0, float (&v)[8]) {
  if (SRC_BF16) {
    const uint4 q = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(row) + k0);
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
    v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
  } else {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(row) + k0);
    const float4 a = __ldcg(p), b = __ldcg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <WeightKind KIND, bool GATE_UP, int NBW>
__global__ void __launch_bounds__(kDecThreads, 1) decode_gemm_kernel(const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.n_stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  uint64_t* redbar = empty + S;  // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(redbar + 2);
  float* red = reinterpret_cast<float*>(smem + 1024);  // [2][warps][16][8]
  uint8_t* stages = smem + 1024 + 2 * kConsumerWarps * kRows * kCols * sizeof(float);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&redbar[0], kConsumerWarps);
    mbar_init(&redbar[1], kConsumerWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const long long n_items = (long long)(*p.n_active) * p.tiles;
  const long long i0 = n_items * blockIdx.x / gridDim.x;
  const long long i1 = n_items * (blockIdx.x + 1) / gridDim.x;
  const int Kh = p.K >> 1;
  const int nb = p.K >> 5;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    long long issued = 0;
    for (long long i = i0; i < i1; ++i, ++issued) {
      if (*abort_flag) break;
      const int stage = (int)(issued % S);
      const long long use = issued / S;
      if (use > 0 && !mbar_wait(&empty[stage], (uint32_t)((use - 1) & 1), p.status)) {
        *abort_flag = 1;
        break;
      }
      const int d = (int)(i / p.tiles), j = (int)(i % p.tiles);
      const int e = p.active[d];
      uint8_t* sw = stages + (size_t)stage * p.stage_bytes;
      uint8_t* ss = sw + kRows * p.row_stride;
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], kRows * (Kh + p.srow_bytes));
      __syncwarp();
      if (lane < kRows) {
        const int row = item_row<GATE_UP>(lane, j, p.I);
        bulk_g2s(sw + lane * p.row_stride, p.w + ((size_t)e * p.N + row) * Kh, Kh, &full[stage], policy);
      } else if (lane == kRows || (GATE_UP && lane == kRows + 1)) {
        const int half = lane - kRows;  // gemm1: 0 gate rows, 1 up rows; gemm2: all 16 rows
        const int rows = GATE_UP ? 8 : kRows;
        const int row0 = item_row<GATE_UP>(half * 8, j, p.I);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws) + ((size_t)e * p.N + row0) * p.srow_bytes;
        bulk_g2s(ss + half * 8 * p.srow_bytes, src, rows * p.srow_bytes, &full[stage], policy);
      }
    }
    // make sure nothing issued is still in flight before the CTA can exit
    const long long first = issued > S ? issued - S : 0;
    for (long long u = first; u < issued; ++u)
      mbar_wait(&full[u % S], (uint32_t)((u / S) & 1), p.status);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int nbw = (nb + kConsumerWarps - 1) / kConsumerWarps;
  const int wb0 = min(nb, warp * nbw), wb1 = min(nb, wb0 + nbw);
  constexpr bool kSrcBf16 = GATE_UP;

  uint32_t xf[NBW][4];
  float inv0 = 1.f, inv1 = 1.f;  // power-of-two undo for accumulator columns 2t, 2t+1
  int cur_e = -1, cur_grp = -1;
  long long use_cnt = 0;  // reduction-buffer uses

  long long it = 0;
  for (long long i = i0; i < i1; ++i, ++it) {
    if (*abort_flag) break;
    const int stage = (int)(it % S);
    const int d = (int)(i / p.tiles), j = (int)(i % p.tiles);
    const int e = p.active[d];
    const int base = p.offsets[e];
    const int npairs = p.offsets[e + 1] - base;
    const int ngroups = (npairs + kCols - 1) / kCols;
    if (!mbar_wait(&full[stage], (uint32_t)((it / S) & 1), p.status)) {
      *abort_flag = 1;
      break;
    }
    const uint8_t* sw = stages + (size_t)stage * p.stage_bytes;
    const uint8_t* ss = sw + kRows * p.row_stride;
    bool stop = false;
    for (int grp = 0; grp < ngroups; ++grp) {
      if (e != cur_e || grp != cur_grp) {
        // ---- activation fragments for pairs grp*8 .. grp*8+7 over this warp's K range
        const int slot = grp * kCols + g;
        const bool valid = slot < npairs;
        const void* row = nullptr;
        if (valid) {
          if (GATE_UP) {
            const int tok = p.sorted_pair[base + slot] / p.topk;
            row = reinterpret_cast<const uint16_t*>(p.src) + (size_t)tok * p.K;
          } else {
            row = reinterpret_cast<const float*>(p.src) + (size_t)(base + slot) * p.K;
          }
        }
        float mx = 0.f;
#pragma unroll
        for (int bb = 0; bb < NBW; ++bb) {
          const int b = wb0 + bb;
          if (valid && b < wb1) {
            float v[8];
            load8<kSrcBf16>(row, b * 32 + 8 * t, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(v[q]));
          }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        int ex = 0;
        if (mx > 0.f) {
          const int lg = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2), normal mx
          ex = min(max(14 - lg, -126), 126);
        }
        const float sc = exp2_int(ex);
#pragma unroll
        for (int bb = 0; bb < NBW; ++bb) {
          const int b = wb0 + bb;
          float v[8];
          if (valid && b < wb1) {
            load8<kSrcBf16>(row, b * 32 + 8 * t, v);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] *= sc;
          if (KIND == WeightKind::kMxfp4) {
            xf[bb][0] = f32x2_to_f16x2(v[0], v[1]);
            xf[bb][1] = f32x2_to_f16x2(v[2], v[3]);
            xf[bb][2] = f32x2_to_f16x2(v[4], v[5]);
            xf[bb][3] = f32x2_to_f16x2(v[6], v[7]);
          } else {
            xf[bb][0] = f32x2_to_f16x2(v[0], v[4]);
            xf[bb][1] = f32x2_to_f16x2(v[1], v[5]);
            xf[bb][2] = f32x2_to_f16x2(v[2], v[6]);
            xf[bb][3] = f32x2_to_f16x2(v[3], v[7]);
          }
        }
        const int ex0 = __shfl_sync(0xffffffffu, ex, (2 * t) * 4);
        const int ex1 = __shfl_sync(0xffffffffu, ex, (2 * t + 1) * 4);
        inv0 = exp2_int(-ex0);
        inv1 = exp2_int(-ex1);
        cur_e = e;
        cur_grp = grp;
      }

      // ---- main loop over this warp's 32-element blocks
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int bb = 0; bb < NBW; ++bb) {
        const int b = wb0 + bb;
        if (b < wb1) {
          const uint8_t* rg = sw + g * p.row_stride + b * 16 + 4 * t;
          const uint32_t wg = *reinterpret_cast<const uint32_t*>(rg);
          const uint32_t wg8 = *reinterpret_cast<const uint32_t*>(rg + 8 * p.row_stride);
          float sg, sg8;
          uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
          if (KIND == WeightKind::kMxfp4) {
            sg = e8m0_to_float(ss[g * p.srow_bytes + b]);
            sg8 = e8m0_to_float(ss[(g + 8) * p.srow_bytes + b]);
            e2m1x8_to_f16x8(wg, a0, a1, a2, a3);
            e2m1x8_to_f16x8(wg8, c0, c1, c2, c3);
          } else {
            const float* sf = reinterpret_cast<const float*>(ss);
            const int spr = p.srow_bytes >> 2;
            sg = sf[g * spr + b];
            sg8 = sf[(g + 8) * spr + b];
            int4x8_to_f16x8(wg, a0, a1, a2, a3);
            int4x8_to_f16x8(wg8, c0, c1, c2, c3);
          }
          float dd[4];
          mma_f16_16816(dd, a0, c0, a1, c1, xf[bb][0], xf[bb][1], zero);
          mma_f16_16816(dd, a2, c2, a3, c3, xf[bb][2], xf[bb][3], dd);
          acc[0] = fmaf(sg, dd[0], acc[0]);
          acc[1] = fmaf(sg, dd[1], acc[1]);
          acc[2] = fmaf(sg8, dd[2], acc[2]);
          acc[3] = fmaf(sg8, dd[3], acc[3]);
        }
      }
      if (grp == ngroups - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }

      // ---- cross-warp reduction and epilogue
      const int buf = (int)(use_cnt & 1);
      float* rb = red + buf * (kConsumerWarps * kRows * kCols);
      float* rw = rb + warp * (kRows * kCols);
      *reinterpret_cast<float2*>(rw + g * kCols + 2 * t) = make_float2(acc[0] * inv0, acc[1] * inv1);
      *reinterpret_cast<float2*>(rw + (g + 8) * kCols + 2 * t) = make_float2(acc[2] * inv0, acc[3] * inv1);
      __syncwarp();
      if (lane == 0) mbar_arrive(&redbar[buf]);
      // every consumer waits: a warp may only write this buffer again two uses
      // later, after all warps have arrived at the use in between
      const bool epi = GATE_UP ? (tid < 64) : (tid < 128);
      if (!mbar_wait(&redbar[buf], (uint32_t)((use_cnt >> 1) & 1), p.status)) {
        *abort_flag = 1;
        stop = true;
      } else if (epi) {
        if (GATE_UP) {
          const int c = tid >> 3, r = tid & 7;
          float hg = 0.f, hu = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            hg += rb[w * kRows * kCols + r * kCols + c];
            hu += rb[w * kRows * kCols + (r + 8) * kCols + c];
          }
          const int slot = grp * kCols + c;
          if (slot < npairs) p.dst[(size_t)(base + slot) * p.I + 8 * j + r] = silu(hg) * hu;
        } else {
          const int c = tid >> 4, r = tid & 15;
          float y = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) y += rb[w * kRows * kCols + r * kCols + c];
          const int slot = grp * kCols + c;
          if (slot < npairs) {
            const int pair = p.sorted_pair[base + slot];
            p.dst[(size_t)pair * p.N + kRows * j + r] = y;
          }
        }
      }
      ++use_cnt;
      if (stop) break;
    }
    if (stop) break;
  }
}

__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ ybuf,
                                                      const int32_t* __restrict__ ids,
                                                      const float* __restrict__ topk_w, int E, int topk,
                                                      int H, uint16_t* __restrict__ out) {
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < topk; ++k) {
    const int pr = t * topk + k;
    const int e = ids[pr];
    if ((unsigned)e >= (unsigned)E) continue;
    const float wk = topk_w[pr];
    const float4 y = __ldcg(reinterpret_cast<const float4*>(ybuf + (size_t)pr * H) + c4);
    acc.x = fmaf(wk, y.x, acc.x);
    acc.y = fmaf(wk, y.y, acc.y);
    acc.z = fmaf(wk, y.z, acc.z);
    acc.w = fmaf(wk, y.w, acc.w);
  }
  uint2 o;
  o.x = f32x2_to_bf16x2(acc.x, acc.y);
  o.y = f32x2_to_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(out + (size_t)t * H + 4 * c4) = o;
}

template <WeightKind KIND, bool GATE_UP, int NBW>
cudaError_t launch_gemm(const GemmParams& gp, int grid, cudaStream_t s) {
  const size_t smem = 1024 + 2 * kConsumerWarps * kRows * kCols * sizeof(float) + (size_t)gp.n_stages * gp.stage_bytes;
  auto kern = decode_gemm_kernel<KIND, GATE_UP, NBW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDecThreads, smem, s>>>(gp);
  return cudaGetLastError();
}

template <WeightKind KIND, bool GATE_UP>
cudaError_t dispatch_nbw(const GemmParams& gp, int grid, cudaStream_t s) {
  const int nbw = ((gp.K >> 5) + kConsumerWarps - 1) / kConsumerWarps;
  if (nbw <= 8) return launch_gemm<KIND, GATE_UP, 8>(gp, grid, s);
  if (nbw <= 16) return launch_gemm<KIND, GATE_UP, 16>(gp, grid, s);
  return launch_gemm<KIND, GATE_UP, 32>(gp, grid, s);
}

void fill_stage_geometry(GemmParams& gp, WeightKind kind) {
  gp.row_stride = (gp.K >> 1) + 16;
  gp.srow_bytes = (gp.K >> 5) * (kind == WeightKind::kMxfp4 ? 1 : 4);
  const int raw = kRows * gp.row_stride + kRows * gp.srow_bytes;
  gp.stage_bytes = (raw + 127) & ~127;
  const int avail = kSmemBudget - 1024 - 2 * kConsumerWarps * kRows * kCols * (int)sizeof(float);
  int st = avail / gp.stage_bytes;
  gp.n_stages = st > 8 ? 8 : st;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  GemmParams g1{};
  g1.w = a.w13;
  g1.ws = a.w13_s;
  g1.N = 2 * a.I;
  g1.K = a.H;
  g1.I = a.I;
  g1.tiles = a.I / 8;
  g1.src = a.x;
  g1.offsets = a.route.offsets;
  g1.active = a.route.active;
  g1.n_active = a.route.n_active;
  g1.sorted_pair = a.route.sorted_pair;
  g1.topk = a.topk;
  g1.dst = a.abuf;
  g1.status = a.status;
  fill_stage_geometry(g1, a.kind);

  GemmParams g2 = g1;
  g2.w = a.w2;
  g2.ws = a.w2_s;
  g2.N = a.H;
  g2.K = a.I;
  g2.tiles = a.H / kRows;
  g2.src = a.abuf;
  g2.dst = a.ybuf;
  fill_stage_geometry(g2, a.kind);
  if (g1.n_stages < 2 || g2.n_stages < 2) return cudaErrorInvalidValue;

  cudaError_t e;
  const bool fp4 = a.kind == WeightKind::kMxfp4;
  timing_mark(1, false, s);
  e = fp4 ? dispatch_nbw<WeightKind::kMxfp4, true>(g1, a.num_sms, s)
          : dispatch_nbw<WeightKind::kInt4, true>(g1, a.num_sms, s);
  timing_mark(1, true, s);
  if (e != cudaSuccess) return e;
  timing_mark(2, false, s);
  e = fp4 ? dispatch_nbw<WeightKind::kMxfp4, false>(g2, a.num_sms, s)
          : dispatch_nbw<WeightKind::kInt4, false>(g2, a.num_sms, s);
  timing_mark(2, true, s);
  if (e != cudaSuccess) return e;
  dim3 cgrid((a.H / 4 + 127) / 128, a.T);
  timing_mark(3, false, s);
  combine_kernel<<<cgrid, 128, 0, s>>>(a.ybuf, a.topk_ids, a.topk_w, a.E, a.topk, a.H,
                                       reinterpret_cast<uint16_t*>(a.out));
  timing_mark(3, true, s);
  return cudaGetLastError();
}

}  // namespace moe
