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
// Grouping: the routing kernel's lists, or for up to 128 pairs a grouping
// every CTA builds itself in shared memory (then no routing kernel runs).
//
// Work unit = (active expert, group of up to 8 of its pairs, 32 weight rows x
// all of K).  For gemm1 the 32 rows are 16 gate rows j..j+15 and the matching
// 16 up rows I+j.., so the activation is local to the unit.  Units are split
// into one contiguous run per CTA (one CTA per SM, persistent); consecutive
// units of one CTA share an expert and group, so its activations stay in
// registers across units.
//
// Per CTA (16 warps): one producer warp streams each unit's 32 weight rows
// (one cp.async.bulk per row into a padded shared-memory stage, so consumer
// reads are bank-conflict-free) and their scales through an mbarrier ring.
// Fourteen consumer warps split K.  Each turns its part of the packed rows into
// m16n8k16 f16 MMA operands (E2M1 pairs via cvt.rn.f16x2.e2m1x2, exact; int4
// pairs via the 1024-offset f16 trick, exact) and multiplies them by up to 8
// activation columns held in registers; the per-32-block weight scale is
// applied to each block's fp32 partial sum (E8M0 pairs decoded with
// cvt.rn.bf16x2.ue8m0x2, exact).  Activations enter the MMA as f16 scaled by a
// power of two per (pair, warp K-range) so they cannot overflow; the scale is
// removed in fp32 afterwards.  The consumer warps hand their partial sums to an
// epilogue warp through a ring of shared-memory buffers; it reduces them and
// writes the results while the consumers go on with the next units.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kConsumerWarps = 14;
constexpr int kProducerWarp = kConsumerWarps;      // streams weights
constexpr int kEpilogueWarp = kConsumerWarps + 1;  // reduces partial sums, writes results
constexpr int kDecThreads = (kConsumerWarps + 2) * 32;
constexpr int kTiles = 2;             // 16-row MMA tiles per item
constexpr int kRows = 16 * kTiles;    // weight rows per item
constexpr int kGroup = 8;             // pair columns per group (one 8-column MMA block)
constexpr int kRedFloats = kConsumerWarps * kRows * kGroup;  // one reduction buffer
constexpr int kRedBufs = 3;                                  // reduction ring depth
static_assert(kGroup == kMoeGroup, "routing and the decode kernels must agree on the group size");
// Batches of at most kLocalRoute pairs are grouped by every CTA itself, in
// shared memory, at the start of both kernels: no routing kernel runs before
// them.  Region: active experts, their first sorted position, their group
// prefix, sorted pairs, count.
constexpr int kLocalRoute = 128;
constexpr int kRouteBytes = 2304;
static_assert(kRouteBytes >= (4 * kLocalRoute + 3) * 4 && kRouteBytes % 256 == 0, "local grouping region");
static_assert(kLocalRoute == kMaxLocalRoutePairs, "api and decode kernels must agree on the local routing limit");
constexpr int kSmemBudget = 226 * 1024;

struct GemmParams {
  const uint8_t* w;        // packed weights [E][N][K/2]
  const void* ws;          // scales [E][N][K/32], u8 (E8M0) or f32
  int N, K, I;             // rows per expert, reduction size, I (gate/up split for gemm1)
  int tiles;               // weight tiles per expert
  const void* src;         // gemm1: x bf16 [T][K]; gemm2: abuf f32 [P][K]
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  const int32_t* gprefix;  // [n_active+1] exclusive prefix of 8-pair groups over active experts
  const int32_t* sorted_pair;
  int topk;
  const int32_t* ids;      // topk ids [P], for grouping inside the kernel
  int E, P;
  int local;               // 1: group the pairs in shared memory (P <= kLocalRoute)
  float* dst;              // gemm1: abuf [P][I]; gemm2: ybuf [P][N]
  uint32_t* status;
  int row_stride;          // bytes between staged weight rows (K/2 + 16)
  int srow_bytes;          // scale bytes per weight row
  int stage_bytes;
  int n_stages;
};

// (c0, c1) += s * (x0, x1) as one packed f32x2 FMA (same rounding as two fmaf).
__device__ __forceinline__ void fma_f32x2_bcast(float& c0, float& c1, float s, float x0, float x1) {
  asm("{\n .reg .b64 d, a, b, c;\n mov.b64 a, {%2, %2};\n mov.b64 b, {%3, %4};\n mov.b64 c, {%0, %1};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(c0), "+f"(c1)
      : "f"(s), "f"(x0), "f"(x1));
}

__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Eight packed int4 (two's complement) -> four f16x2, pairs (i, i+4), exact.
// With n = q + 8 (offset binary), n placed in the low mantissa bits of f16
// 1024 gives 1024 + n (minus 1032: q); n placed 4 bits higher gives 1024 + 16n
// (times 1/16 minus 72: q); one byte permute brings nibbles 2, 3, 6, 7 down.
__device__ __forceinline__ void int4x8_to_f16x8(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
  const uint32_t u = w ^ 0x88888888u;   // offset binary: q + 8
  const uint32_t v = prmt(u, 0u, 0x4341u);  // bytes 1 and 3 of u into bytes 0 and 2
  const uint32_t magic = 0x64006400u;   // f16 1024 in both halves
  const uint32_t bias = 0x64086408u;    // f16 1032
  const uint32_t sixteenth = 0x2C002C00u;  // f16 1/16
  const uint32_t m72 = 0xD480D480u;     // f16 -72
  o0 = f16x2_sub((u & 0x000F000Fu) | magic, bias);
  o1 = f16x2_fma((u & 0x00F000F0u) | magic, sixteenth, m72);
  o2 = f16x2_sub((v & 0x000F000Fu) | magic, bias);
  o3 = f16x2_fma((v & 0x00F000F0u) | magic, sixteenth, m72);
}

// Two E8M0 bytes (low byte = first) -> their values 2^(s-127) as floats, exact
// (bf16 keeps the full exponent range, including 2^-127).
__device__ __forceinline__ void e8m0x2_to_float2(uint32_t two_bytes, float& lo, float& hi) {
  uint32_t r;
  asm("{\n .reg .b16 b;\n cvt.u16.u32 b, %1;\n cvt.rn.bf16x2.ue8m0x2 %0, b;\n}" : "=r"(r) : "r"(two_bytes));
  lo = __uint_as_float(r << 16);
  hi = __uint_as_float(r & 0xFFFF0000u);
}

template <bool GATE_UP>
__device__ __forceinline__ int item_row(int r, int j, int I) {
  if (GATE_UP) return r < kRows / 2 ? (kRows / 2) * j + r : I + (kRows / 2) * j + (r - kRows / 2);
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

// Activation fragments of one 8-pair column block (pairs slot0 + g, g = lane/4)
// over the calling warp's blocks [wb0, wb0 + cnt), as f16 scaled by a power of
// two per pair; inv receives the undo factors for accumulator columns 2t, 2t+1.
template <WeightKind KIND, bool GATE_UP, int NBW>
__device__ __forceinline__ void load_frags(const GemmParams& p, const int32_t* spair, int slot0, int base, int npairs,
                                           int wb0, int cnt, int g, int t, uint32_t (&xf)[NBW][4], float (&inv)[2]) {
  const int slot = slot0 + g;
  const bool valid = slot < npairs;
  const void* row = nullptr;
  if (valid) {
    if (GATE_UP) {
      const int tok = spair[base + slot] / p.topk;
      row = reinterpret_cast<const uint16_t*>(p.src) + (size_t)tok * p.K;
    } else {
      row = reinterpret_cast<const float*>(p.src) + (size_t)(base + slot) * p.K;
    }
  }
  float mx = 0.f;
#pragma unroll
  for (int bb = 0; bb < NBW; ++bb) {
    if (valid && bb < cnt) {
      float v[8];
      load8<GATE_UP>(row, (wb0 + bb) * 32 + 8 * t, v);
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
    float v[8];
    if (valid && bb < cnt) {
      load8<GATE_UP>(row, (wb0 + bb) * 32 + 8 * t, v);
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
  inv[0] = exp2_int(-ex0);
  inv[1] = exp2_int(-ex1);
}

// Scales of rows r and r+8 of one 16-row tile for blocks b, b+1 (b even).
template <WeightKind KIND>
__device__ __forceinline__ void load_scales2(const uint8_t* ss, int srow, int r, int b, float (&s)[2][2]) {
  if (KIND == WeightKind::kMxfp4) {
    const uint32_t u0 = *reinterpret_cast<const uint16_t*>(ss + r * srow + b);
    const uint32_t u1 = *reinterpret_cast<const uint16_t*>(ss + (r + 8) * srow + b);
    e8m0x2_to_float2(u0, s[0][0], s[0][1]);
    e8m0x2_to_float2(u1, s[1][0], s[1][1]);
  } else {
    const float2 f0 = *reinterpret_cast<const float2*>(ss + r * srow + 4 * b);
    const float2 f1 = *reinterpret_cast<const float2*>(ss + (r + 8) * srow + 4 * b);
    s[0][0] = f0.x; s[0][1] = f0.y; s[1][0] = f1.x; s[1][1] = f1.y;
  }
}

template <WeightKind KIND>
__device__ __forceinline__ void weights_to_f16(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  if (KIND == WeightKind::kMxfp4) e2m1x8_to_f16x8(w, o0, o1, o2, o3);
  else int4x8_to_f16x8(w, o0, o1, o2, o3);
}

// Position in a contiguous run of work units (active expert d, 8-pair group
// grp, weight tile j), advanced without divisions (one at the start).
struct UnitCursor {
  int d, grp, j, end;  // end = first unit of expert d + 1
  __device__ __forceinline__ void init(const int32_t* gpre, int tiles, int d0, int u0) {
    d = d0;
    const int rem = u0 - gpre[d] * tiles;
    grp = rem / tiles;
    j = rem - grp * tiles;
    end = gpre[d + 1] * tiles;
  }
  // step to unit u_next (= the current unit + 1); call only for u_next < the run's end
  __device__ __forceinline__ void next(const int32_t* gpre, int tiles, int u_next) {
    if (++j == tiles) {
      j = 0;
      ++grp;
    }
    if (u_next == end) {  // every active expert has at least one unit
      ++d;
      grp = 0;
      j = 0;
      end = gpre[d + 1] * tiles;
    }
  }
};

template <WeightKind KIND, bool GATE_UP, int NBW>
__global__ void __launch_bounds__(kDecThreads, 1) decode_gemm_kernel(const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.n_stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  uint64_t* red_full = empty + S;            // [kRedBufs]
  uint64_t* red_empty = red_full + kRedBufs;  // [kRedBufs]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red_empty + kRedBufs);
  int32_t* r_act = reinterpret_cast<int32_t*>(smem + 1024);  // local grouping, see kLocalRoute
  int32_t* r_base = r_act + kLocalRoute;
  int32_t* r_gpre = r_base + kLocalRoute + 1;
  int32_t* r_pair = r_gpre + kLocalRoute + 1;
  int32_t* r_n = r_pair + kLocalRoute;
  float* red = reinterpret_cast<float*>(smem + 1024 + kRouteBytes);  // [kRedBufs][warps][32 rows][8 pair columns]
  uint8_t* stages = smem + 1024 + kRouteBytes + kRedBufs * kRedFloats * sizeof(float);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < kRedBufs; ++b) {
      mbar_init(&red_full[b], kConsumerWarps);
      mbar_init(&red_empty[b], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // gate_up reads the grouping of the kernel before it; down reads only
  // weights and grouping here and waits for gate_up's activations further down
  if (GATE_UP) grid_dep_wait();
  grid_dep_launch_dependents();

  if (p.local) {
    // Group the P <= kLocalRoute pairs by expert: stable order (expert
    // ascending, pair index ascending), active experts ascending, 8-pair
    // groups per active expert.  Scratch lives in the weight stages, which
    // nothing uses yet.
    int32_t* ids_s = reinterpret_cast<int32_t*>(stages);       // [P] expert or -1
    int32_t* first_g = ids_s + kLocalRoute;                    // [P] groups of its expert at its first pair, else 0
    const int P = p.P;
    if (tid < P) {
      const int e = p.ids[tid];
      ids_s[tid] = (unsigned)e < (unsigned)p.E ? e : -1;
    }
    __syncthreads();
    int e = -1, less = 0, rank = 0, cnt = 0;
    if (tid < P) {
      e = ids_s[tid];
      if (e >= 0) {
        for (int q = 0; q < P; ++q) {
          const int f = ids_s[q];
          less += (f >= 0 && f < e) ? 1 : 0;
          cnt += f == e ? 1 : 0;
          rank += (f == e && q < tid) ? 1 : 0;
        }
      }
      first_g[tid] = (e >= 0 && rank == 0) ? (cnt + kGroup - 1) / kGroup : 0;
    }
    __syncthreads();
    if (tid < P && e >= 0) {
      r_pair[less + rank] = tid;
      if (rank == 0) {
        int dd = 0, gp = 0;
        for (int q = 0; q < P; ++q) {
          const int fg = first_g[q];
          if (fg > 0 && ids_s[q] < e) {
            ++dd;
            gp += fg;
          }
        }
        r_act[dd] = e;
        r_base[dd] = less;
        r_gpre[dd] = gp;
      }
    }
    if (tid == 0) {
      int n = 0, tot = 0, gt = 0;
      for (int q = 0; q < P; ++q) {
        if (first_g[q] > 0) {
          ++n;
          gt += first_g[q];
        }
        if (ids_s[q] >= 0) ++tot;
      }
      r_base[n] = tot;
      r_gpre[n] = gt;
      *r_n = n;
    }
    __syncthreads();
  }
  // grouping views: shared memory (indexed by active expert) or the routing
  // kernel's output (offsets indexed by expert id)
  const bool local = p.local != 0;
  const int32_t* act = local ? r_act : p.active;
  const int32_t* gpre = local ? r_gpre : p.gprefix;
  const int32_t* spair = local ? r_pair : p.sorted_pair;

  // Work units: (active expert d, 8-pair group, weight tile j), group-major
  // within an expert, so a CTA's contiguous run reloads activations only at
  // group boundaries.  Experts with more than 8 pairs stream their weights
  // once per group.
  const int n_act = local ? *r_n : *p.n_active;
  const int n_units = gpre[n_act] * p.tiles;
  const int u0 = (int)((long long)n_units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)n_units * (blockIdx.x + 1) / gridDim.x);
  const int Kh = p.K >> 1;
  const int nb = p.K >> 5;
  // first active expert whose units reach u0
  int d0 = 0;
  {
    int lo = 0, hi = n_act;  // largest d with gprefix[d] * tiles <= u0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (gpre[mid] * p.tiles <= u0) lo = mid; else hi = mid;
    }
    d0 = lo;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    int issued = 0, stage = 0;
    uint32_t phase = 0;
    UnitCursor cur;
    if (u0 < u1) cur.init(gpre, p.tiles, d0, u0);
    for (int u = u0; u < u1; ++u, ++issued) {
      if (*abort_flag) break;
      if (u > u0) cur.next(gpre, p.tiles, u);
      const int j = cur.j;
      if (issued >= S && !mbar_wait(&empty[stage], phase ^ 1u, p.status)) {
        *abort_flag = 1;
        break;
      }
      const int e = act[cur.d];
      uint8_t* sw = stages + (size_t)stage * p.stage_bytes;
      uint8_t* ss = sw + kRows * p.row_stride;
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], kRows * (Kh + p.srow_bytes));
      __syncwarp();
      {
        const int row = item_row<GATE_UP>(lane, j, p.I);
        bulk_g2s(sw + lane * p.row_stride, p.w + ((size_t)e * p.N + row) * Kh, Kh, &full[stage], policy);
      }
      if (lane < (GATE_UP ? 2 : 1)) {
        // scales: gemm1 gate rows then up rows (each contiguous); gemm2 all rows
        const int rows = GATE_UP ? kRows / 2 : kRows;
        const int row0 = item_row<GATE_UP>(lane * (kRows / 2), j, p.I);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws) + ((size_t)e * p.N + row0) * p.srow_bytes;
        bulk_g2s(ss + lane * (kRows / 2) * p.srow_bytes, src, rows * p.srow_bytes, &full[stage], policy);
      }
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // make sure nothing issued is still in flight before the CTA can exit:
    // wait for the last min(issued, S) fills, walking the ring backwards
    for (int v = 0; v < (issued < S ? issued : S); ++v) {
      if (stage == 0) {
        stage = S - 1;
        phase ^= 1u;
      } else {
        --stage;
      }
      mbar_wait(&full[stage], phase, p.status);
    }
    return;
  }

  if (warp == kEpilogueWarp) {
    // ------------------------------------------------------------ epilogue
    // Sums the consumer warps' partials of each unit and writes the results,
    // while the consumers already work on the next units.
    int rbuf = 0;
    uint32_t rph = 0;
    UnitCursor cur;
    if (u0 < u1) cur.init(gpre, p.tiles, d0, u0);
    for (int u = u0; u < u1; ++u) {
      if (u > u0) cur.next(gpre, p.tiles, u);
      const int d = cur.d, grp = cur.grp, j = cur.j;
      const int e = act[d];
      const int base = local ? r_base[d] : p.offsets[e];
      const int npairs = (local ? r_base[d + 1] : p.offsets[e + 1]) - base;
      if (!mbar_wait(&red_full[rbuf], rph, p.status)) {
        *abort_flag = 1;
        break;
      }
      const float* rb = red + rbuf * kRedFloats;
      if (GATE_UP) {
        constexpr int kOut = kRows / 2;  // activated outputs per unit
#pragma unroll
        for (int q = 0; q < kOut * kGroup / 32; ++q) {
          const int idx = lane + 32 * q;
          const int r = idx / kGroup, c = idx % kGroup;
          float hg = 0.f, hu = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            hg += rb[w * kRows * kGroup + r * kGroup + c];
            hu += rb[w * kRows * kGroup + (r + kOut) * kGroup + c];
          }
          const int slot = grp * kGroup + c;
          if (slot < npairs) p.dst[(size_t)(base + slot) * p.I + kOut * j + r] = silu(hg) * hu;
        }
      } else {
#pragma unroll
        for (int q = 0; q < kRows * kGroup / 32; ++q) {
          const int idx = lane + 32 * q;
          const int r = idx / kGroup, c = idx % kGroup;
          float y = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) y += rb[w * kRows * kGroup + r * kGroup + c];
          const int slot = grp * kGroup + c;
          if (slot < npairs) {
            const int pair = spair[base + slot];
            p.dst[(size_t)pair * p.N + kRows * j + r] = y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[rbuf]);
      if (++rbuf == kRedBufs) {
        rbuf = 0;
        rph ^= 1u;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  // even number of blocks per warp, so blocks are processed in pairs
  const int nbw = 2 * ((nb + 2 * kConsumerWarps - 1) / (2 * kConsumerWarps));
  const int wb0 = min(nb, warp * nbw);
  const int cnt = min(nbw, nb - wb0);

  uint32_t xf[NBW][4];
  float inv[2];  // power-of-two undo for accumulator columns 2t, 2t+1
  int cur_e = -1, cur_grp = -1;
  if (!GATE_UP) grid_dep_wait();  // the activations come from the gate_up kernel

  int it = 0, stage = 0, rbuf = 0;
  uint32_t phase = 0, rph = 0;
  UnitCursor cur;
  if (u0 < u1) cur.init(gpre, p.tiles, d0, u0);
  for (int u = u0; u < u1; ++u, ++it) {
    if (*abort_flag) break;
    if (u > u0) cur.next(gpre, p.tiles, u);
    const int d = cur.d, grp = cur.grp;
    const int e = act[d];
    const int base = local ? r_base[d] : p.offsets[e];
    const int npairs = (local ? r_base[d + 1] : p.offsets[e + 1]) - base;
    if (e != cur_e || grp != cur_grp) {
      load_frags<KIND, GATE_UP, NBW>(p, spair, grp * kGroup, base, npairs, wb0, cnt, g, t, xf, inv);
      cur_e = e;
      cur_grp = grp;
    }
    if (!mbar_wait(&full[stage], phase, p.status)) {
      *abort_flag = 1;
      break;
    }
    const uint8_t* sw = stages + (size_t)stage * p.stage_bytes;
    const uint8_t* ss = sw + kRows * p.row_stride;

    // ---- main loop over this warp's 32-element blocks, two at a time
    float acc[kTiles][4];
#pragma unroll
    for (int tl = 0; tl < kTiles; ++tl) acc[tl][0] = acc[tl][1] = acc[tl][2] = acc[tl][3] = 0.f;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int bb = 0; bb < NBW; bb += 2) {
      if (bb < cnt) {
        const int b = wb0 + bb;
#pragma unroll
        for (int tl = 0; tl < kTiles; ++tl) {
          const int r = 16 * tl + g;
          float sc[2][2];  // [row r / r+8][block b / b+1]
          load_scales2<KIND>(ss, p.srow_bytes, r, b, sc);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint8_t* rg = sw + r * p.row_stride + (b + h) * 16 + 4 * t;
            uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
            weights_to_f16<KIND>(*reinterpret_cast<const uint32_t*>(rg), a0, a1, a2, a3);
            weights_to_f16<KIND>(*reinterpret_cast<const uint32_t*>(rg + 8 * p.row_stride), c0, c1, c2, c3);
            float dd[4];
            mma_f16_16816(dd, a0, c0, a1, c1, xf[bb + h][0], xf[bb + h][1], zero);
            mma_f16_16816(dd, a2, c2, a3, c3, xf[bb + h][2], xf[bb + h][3], dd);
            fma_f32x2_bcast(acc[tl][0], acc[tl][1], sc[0][h], dd[0], dd[1]);
            fma_f32x2_bcast(acc[tl][2], acc[tl][3], sc[1][h], dd[2], dd[3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }

    // ---- hand the partial sums to the epilogue warp
    if (it >= kRedBufs && !mbar_wait(&red_empty[rbuf], rph ^ 1u, p.status)) {
      *abort_flag = 1;
      break;
    }
    float* rw = red + rbuf * kRedFloats + warp * (kRows * kGroup);
#pragma unroll
    for (int tl = 0; tl < kTiles; ++tl) {
      const int r = 16 * tl + g;
      *reinterpret_cast<float2*>(rw + r * kGroup + 2 * t) = make_float2(acc[tl][0] * inv[0], acc[tl][1] * inv[1]);
      *reinterpret_cast<float2*>(rw + (r + 8) * kGroup + 2 * t) =
          make_float2(acc[tl][2] * inv[0], acc[tl][3] * inv[1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&red_full[rbuf]);
    if (++rbuf == kRedBufs) {
      rbuf = 0;
      rph ^= 1u;
    }
  }
}

__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ ybuf,
                                                      const int32_t* __restrict__ ids,
                                                      const float* __restrict__ topk_w, int E, int topk,
                                                      int H, uint16_t* __restrict__ out) {
  __shared__ int s_ids[64];
  __shared__ float s_w[64];
  // the next kernel on the stream may start its prologue now; it waits
  // (griddepcontrol.wait) for this grid to complete before using anything
  grid_dep_launch_dependents();
  grid_dep_wait();  // ybuf comes from the down kernel
  const int t = blockIdx.y;
  if (threadIdx.x < topk) {
    s_ids[threadIdx.x] = ids[t * topk + threadIdx.x];
    s_w[threadIdx.x] = topk_w[t * topk + threadIdx.x];
  }
  __syncthreads();
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* yb = reinterpret_cast<const float4*>(ybuf + (size_t)t * topk * H) + c4;
  const int h4 = H / 4;
  for (int k0 = 0; k0 < topk; k0 += 8) {
    float4 y[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool valid = k0 + k < topk && (unsigned)s_ids[k0 + k] < (unsigned)E;
      y[k] = valid ? __ldcg(yb + (size_t)(k0 + k) * h4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k0 + k < topk && (unsigned)s_ids[k0 + k] < (unsigned)E) {
        const float wk = s_w[k0 + k];
        acc.x = fmaf(wk, y[k].x, acc.x);
        acc.y = fmaf(wk, y[k].y, acc.y);
        acc.z = fmaf(wk, y[k].z, acc.z);
        acc.w = fmaf(wk, y[k].w, acc.w);
      }
    }
  }
  uint2 o;
  o.x = f32x2_to_bf16x2(acc.x, acc.y);
  o.y = f32x2_to_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(out + (size_t)t * H + 4 * c4) = o;
}

template <WeightKind KIND, bool GATE_UP, int NBW>
cudaError_t launch_gemm(const GemmParams& gp, int grid, cudaStream_t s) {
  const size_t smem = 1024 + kRouteBytes + kRedBufs * kRedFloats * sizeof(float) + (size_t)gp.n_stages * gp.stage_bytes;
  auto kern = decode_gemm_kernel<KIND, GATE_UP, NBW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(kDecThreads), smem, s, true, gp);
}

template <WeightKind KIND, bool GATE_UP>
cudaError_t dispatch_nbw(const GemmParams& gp, int grid, cudaStream_t s) {
  const int nbw = 2 * (((gp.K >> 5) + 2 * kConsumerWarps - 1) / (2 * kConsumerWarps));
  if (nbw <= 8) return launch_gemm<KIND, GATE_UP, 8>(gp, grid, s);
  if (nbw <= 16) return launch_gemm<KIND, GATE_UP, 16>(gp, grid, s);
  if (nbw <= 24) return launch_gemm<KIND, GATE_UP, 24>(gp, grid, s);
  return launch_gemm<KIND, GATE_UP, 38>(gp, grid, s);
}

void fill_stage_geometry(GemmParams& gp, WeightKind kind) {
  gp.row_stride = (gp.K >> 1) + 16;
  gp.srow_bytes = (gp.K >> 5) * (kind == WeightKind::kMxfp4 ? 1 : 4);
  const int raw = kRows * gp.row_stride + kRows * gp.srow_bytes;
  gp.stage_bytes = (raw + 127) & ~127;
  const int avail = kSmemBudget - 1024 - kRouteBytes - kRedBufs * kRedFloats * (int)sizeof(float);
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
  g1.tiles = a.I / (kRows / 2);
  g1.src = a.x;
  g1.offsets = a.route.offsets;
  g1.active = a.route.active;
  g1.n_active = a.route.n_active;
  g1.gprefix = a.route.gprefix;
  g1.sorted_pair = a.route.sorted_pair;
  g1.topk = a.topk;
  g1.ids = a.topk_ids;
  g1.E = a.E;
  g1.P = a.T * a.topk;
  g1.local = g1.P <= kLocalRoute ? 1 : 0;
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
  e = launch_kernel(combine_kernel, cgrid, dim3(128), 0, s, true, (const float*)a.ybuf, a.topk_ids, a.topk_w, a.E,
                    a.topk, a.H, reinterpret_cast<uint16_t*>(a.out));
  timing_mark(3, true, s);
  return e;
}

}  // namespace moe
