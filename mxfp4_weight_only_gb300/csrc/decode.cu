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
// reduction ring depth: two buffers keep the consumers ahead of the epilogue
// warp (whose per-unit work is short) and leave room for a third weight stage
// of int4 with bf16 scales (65 KB stages; with three buffers only two fit:
// int4 bf16-scale decode 6-7 % slower, the other kinds unchanged)
constexpr int kRedBufs = 2;
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
  uint32_t* epoch;         // fused kernel: call counter and one publication flag per CTA
  uint32_t* flags;
  int row_stride;          // bytes between staged weight rows (K/2 + 16)
  int srow_bytes;          // scale bytes per weight row
  int stage_bytes;
  int n_stages;
  uint64_t wait_ns;        // limit of every bounded wait
  int wait_extra;          // fused kernel, tests only: CTAs its cross-CTA wait expects beyond the grid
  const float* topk_w;     // [T][topk]
  // optional inputs
  const uint16_t* bias;    // bf16 [E][N] added to the outputs (gate_up: b13, down: b2), or null
  const int32_t* emap;     // global -> local expert ids, or null
  int G;                   // entries of emap
  int rwi;                 // router weight on the input (gate_up scales h), unweighted combine
  int aq;                  // activation quantisation of this GEMM's input (ActQuant)
  float ascale;            // kActFp8: the input's static scale, applied to the reduced float32 sums
  float clamp;             // gate_up: outputs clamped to [-clamp, clamp] before the gating (0: off)
};

// (c0, c1) += (s0, s1) * (x0, x1) as one packed f32x2 FMA (same rounding as two fmaf).
__device__ __forceinline__ void fma_f32x2(float& c0, float& c1, float s0, float s1, float x0, float x1) {
  asm("{\n .reg .b64 d, a, b, c;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%0, %1};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(c0), "+f"(c1)
      : "f"(s0), "f"(s1), "f"(x0), "f"(x1));
}

// (d0, d1) = s * (x0, x1) as one packed f32x2 multiply.
__device__ __forceinline__ void mul_f32x2_bcast(float& d0, float& d1, float s, float x0, float x1) {
  asm("{\n .reg .b64 d, a, b;\n mov.b64 a, {%2, %2};\n mov.b64 b, {%3, %4};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d0), "=f"(d1)
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
// Flipping a nibble's top bit (q -> q + 8) and setting the exponent bits of
// 1024 touch disjoint bits of the masked word, so (w & mask) ^ (flip | 1024)
// does both in one logic operation.
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(b), "r"(c));  // (a & b) ^ c
  return r;
}

__device__ __forceinline__ void int4x8_to_f16x8(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
  const uint32_t v = prmt(w, 0u, 0x4341u);  // bytes 1 and 3 of w into bytes 0 and 2
  const uint32_t lo = 0x64086408u;          // f16 1024 | the flip of the low nibble's top bit (bit 3)
  const uint32_t hi = 0x64806480u;          // f16 1024 | the flip of the high nibble's top bit (bit 7)
  const uint32_t bias = 0x64086408u;        // f16 1032
  const uint32_t sixteenth = 0x2C002C00u;   // f16 1/16
  const uint32_t m72 = 0xD480D480u;         // f16 -72
  o0 = f16x2_sub(and_xor(w, 0x000F000Fu, lo), bias);
  o1 = f16x2_fma(and_xor(w, 0x00F000F0u, hi), sixteenth, m72);
  o2 = f16x2_sub(and_xor(v, 0x000F000Fu, lo), bias);
  o3 = f16x2_fma(and_xor(v, 0x00F000F0u, hi), sixteenth, m72);
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

// Converts this lane's activation values over the warp's blocks into f16
// MMA fragments at scale ``sc`` (SCALED) or 1; FIND_MAX also returns their
// largest magnitude (before any quantisation).
template <WeightKind KIND, bool GATE_UP, int NBW, int AQ, bool SCALED, bool FIND_MAX>
__device__ __forceinline__ void convert_frags(const GemmParams& p, const void* row, bool valid, int wb0, int cnt,
                                              int t, float sc, uint32_t (&xf)[NBW][4], float& mx) {
#pragma unroll
  for (int bb = 0; bb < NBW; ++bb) {
    float v[8];
    if (valid && bb < cnt) {
      load8<GATE_UP>(row, (wb0 + bb) * 32 + 8 * t, v);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = 0.f;
    }
    if (FIND_MAX) {
#pragma unroll
      for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(v[q]));
    }
    if (AQ != kActNone) act_quant8(AQ, p.ascale, v);  // warp-uniform: every lane calls it
    if (SCALED) {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] *= sc;
    }
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
}

// Activation fragments of one 8-pair column block (pairs slot0 + g, g = lane/4)
// over the calling warp's blocks [wb0, wb0 + cnt), as f16 scaled by a power of
// two per pair; inv receives the undo factors for accumulator columns 2t, 2t+1.
// One pass converts at scale 1 and finds each range's largest magnitude; only
// when some range of the warp needs a power of two other than 1 does a second
// pass convert again (one global-memory round trip in the common case).
// AQ: the activation quantisation the kernel variant applies (ActQuant, a
// compile-time mode, so each variant carries only its own quantiser and the
// plain variant none).
template <WeightKind KIND, bool GATE_UP, int NBW, int AQ>
__device__ __forceinline__ void load_frags(const GemmParams& p, const int32_t* spair, int slot0, int base, int npairs,
                                           int wb0, int cnt, int g, int t, uint32_t (&xf)[NBW][4], float (&inv)[2]) {
  const int slot = slot0 + g;
  const bool valid = slot < npairs;
  const void* row = nullptr;
  if (valid) {
    if (GATE_UP) {
      const int tok = chk(spair[chk(base + slot, p.P, p.status)], p.P, p.status) / p.topk;
      row = reinterpret_cast<const uint16_t*>(p.src) + (size_t)tok * p.K;
    } else {
      row = reinterpret_cast<const float*>(p.src) + (size_t)chk(base + slot, p.P, p.status) * p.K;
    }
  }
  float mx = 0.f;
  convert_frags<KIND, GATE_UP, NBW, AQ, false, true>(p, row, valid, wb0, cnt, t, 1.f, xf, mx);
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  // power of two taking the range's largest magnitude into [2^14, 2^15) --
  // or 1 when it already lies in [2^-4, 2^15), and the kernel skips the undo
  // multiplies.  Unscaled, values of 2^-14 and more keep f16's 11 bits (bf16
  // inputs from 2^-17 on are exact) and smaller ones are rounded to the f16
  // subnormal grid, an error of at most 2^-25 each: summed over a K of 4096,
  // 2^-9 of the range's largest value.
  //
  // Quantised activations (p.aq): MXFP4 values code * 2^(s-127) are at most
  // 6/5 of their block's largest magnitude, so the same power of two keeps
  // them below 2^15 * 1.2 (finite in f16); FP8 leaves the e4m3 values (exact
  // in f16, at most 448) unscaled.
  int ex = 0;
  if (mx > 0.f && AQ != kActFp8) {
    const int lg = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2), normal mx
    ex = (lg >= -4 && lg <= 14) ? 0 : min(max(14 - lg, -126), 126);
  }
  if (__any_sync(0xffffffffu, ex != 0)) {
    float unused = 0.f;
    convert_frags<KIND, GATE_UP, NBW, AQ, true, false>(p, row, valid, wb0, cnt, t, exp2_int(ex), xf, unused);
  }
  const int ex0 = __shfl_sync(0xffffffffu, ex, (2 * t) * 4);
  const int ex1 = __shfl_sync(0xffffffffu, ex, (2 * t + 1) * 4);
  inv[0] = exp2_int(-ex0);
  inv[1] = exp2_int(-ex1);
  // (FP8: ex is 0 and inv 1; the static scale multiplies the reduced sums in
  // the epilogue, once per output, so the main loop needs no folded scales)
}

// Scales of rows r and r+8 of one 16-row tile for blocks b, b+1 (b even).
template <WeightKind KIND>
__device__ __forceinline__ void load_scales2(const uint8_t* ss, int srow, int r, int b, float (&s)[2][2],
                                             uint32_t* status) {
  if (KIND == WeightKind::kMxfp4) {
    const uint32_t u0 = *reinterpret_cast<const uint16_t*>(ss + r * srow + b);
    const uint32_t u1 = *reinterpret_cast<const uint16_t*>(ss + (r + 8) * srow + b);
    chk_e8m0(u0 | (u1 << 16), 4, status);
    e8m0x2_to_float2(u0, s[0][0], s[0][1]);
    e8m0x2_to_float2(u1, s[1][0], s[1][1]);
  } else if (KIND == WeightKind::kInt4) {
    const float2 f0 = *reinterpret_cast<const float2*>(ss + r * srow + 4 * b);
    const float2 f1 = *reinterpret_cast<const float2*>(ss + (r + 8) * srow + 4 * b);
    s[0][0] = f0.x; s[0][1] = f0.y; s[1][0] = f1.x; s[1][1] = f1.y;
  } else {
    // bfloat16 scales: a bf16 value is the high half of its float
    const uint32_t u0 = *reinterpret_cast<const uint32_t*>(ss + r * srow + 2 * b);
    const uint32_t u1 = *reinterpret_cast<const uint32_t*>(ss + (r + 8) * srow + 2 * b);
    s[0][0] = bf16_lo(u0); s[0][1] = bf16_hi(u0); s[1][0] = bf16_lo(u1); s[1][1] = bf16_hi(u1);
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

// ------------------------------------------------------------------ per-CTA state

constexpr int kMaxStages = 8;  // weight stages at most (fill_stage_geometry caps the count)

// Shared-memory carve-up used by both decode kernels: barriers and flags in
// the first 1 KiB, the local grouping, the reduction ring, the weight stages.
struct CtaSmem {
  uint64_t* full;       // [kMaxStages] weight stage filled
  uint64_t* empty;      // [kMaxStages] weight stage released by every consumer warp
  uint64_t* red_full;   // [kRedBufs] partial sums of one unit handed in by every consumer warp
  uint64_t* red_empty;  // [kRedBufs] reduction buffer drained by the epilogue warp
  volatile int* abort_flag;
  uint32_t* token;      // fused kernel: the value this call publishes
  int32_t* r_act;       // local grouping (batches of at most kLocalRoute pairs)
  int32_t* r_base;
  int32_t* r_gpre;
  int32_t* r_pair;
  int32_t* r_n;
  float* red;           // [kRedBufs][warps][32 rows][8 pair columns]
  uint8_t* stages;
};

__device__ __forceinline__ CtaSmem carve_smem(uint8_t* smem) {
  CtaSmem c;
  c.full = reinterpret_cast<uint64_t*>(smem);
  c.empty = c.full + kMaxStages;
  c.red_full = c.empty + kMaxStages;
  c.red_empty = c.red_full + kRedBufs;
  c.abort_flag = reinterpret_cast<volatile int*>(c.red_empty + kRedBufs);
  c.token = reinterpret_cast<uint32_t*>(c.red_empty + kRedBufs) + 1;
  c.r_act = reinterpret_cast<int32_t*>(smem + 1024);
  c.r_base = c.r_act + kLocalRoute;
  c.r_gpre = c.r_base + kLocalRoute + 1;
  c.r_pair = c.r_gpre + kLocalRoute + 1;
  c.r_n = c.r_pair + kLocalRoute;
  c.red = reinterpret_cast<float*>(smem + 1024 + kRouteBytes);
  c.stages = smem + 1024 + kRouteBytes + kRedBufs * kRedFloats * sizeof(float);
  return c;
}
static_assert((2 * kMaxStages + 2 * kRedBufs) * 8 + 8 <= 1024, "barrier region");
constexpr int kSmemFixed = 1024 + kRouteBytes + kRedBufs * kRedFloats * (int)sizeof(float);

__device__ __forceinline__ void init_barriers(const CtaSmem& c, int S) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], kConsumerWarps);
    }
    for (int b = 0; b < kRedBufs; ++b) {
      mbar_init(&c.red_full[b], kConsumerWarps);
      mbar_init(&c.red_empty[b], 1);
    }
    *c.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
}

// Group the P <= kLocalRoute pairs by expert (whole CTA): stable order (expert
// ascending, pair index ascending), active experts ascending, 8-pair groups
// per active expert.  Scratch lives in the weight stages, which nothing uses
// yet.  Ends with a CTA barrier.
__device__ void local_grouping(const GemmParams& p, const CtaSmem& c) {
  const int tid = threadIdx.x;
  if (p.P <= 32) {
    // one warp holds every pair (lane = pair): ranks among equal experts by
    // __match_any_sync, sorted positions and active-list fields by one pass of
    // shuffles over the 32 lanes; no CTA-wide barrier until the end
    if (tid < 32) {
      const int lane = tid;
      const int e = lane < p.P ? local_expert(p.ids, lane, p.emap, p.G, p.E) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int cnt = __popc(peers);
      const bool first = e >= 0 && rank == 0;
      const int groups = first ? (cnt + kGroup - 1) / kGroup : 0;
      int less = 0, dd = 0, gp = 0;  // valid pairs, active experts and their groups with a smaller id
#pragma unroll 8
      for (int q = 0; q < 32; ++q) {
        const int f = __shfl_sync(0xffffffffu, e, q);
        const int fg = __shfl_sync(0xffffffffu, groups, q);
        const bool smaller = f >= 0 && f < e;
        less += smaller ? 1 : 0;
        dd += (smaller && fg > 0) ? 1 : 0;
        gp += smaller ? fg : 0;
      }
      if (e >= 0) c.r_pair[less + rank] = lane;
      if (first) {
        c.r_act[dd] = e;
        c.r_base[dd] = less;
        c.r_gpre[dd] = gp;
      }
      const int n = __popc(__ballot_sync(0xffffffffu, first));
      const int tot = __popc(__ballot_sync(0xffffffffu, e >= 0));
      int gt = groups;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gt += __shfl_xor_sync(0xffffffffu, gt, o);
      if (lane == 0) {
        c.r_base[n] = tot;
        c.r_gpre[n] = gt;
        *c.r_n = n;
      }
    }
    __syncthreads();
    return;
  }
  int32_t* ids_s = reinterpret_cast<int32_t*>(c.stages);  // [P] expert or -1
  int32_t* first_g = ids_s + kLocalRoute;                 // [P] groups of its expert at its first pair, else 0
  const int P = p.P;
  if (tid < P) ids_s[tid] = local_expert(p.ids, tid, p.emap, p.G, p.E);
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
    c.r_pair[less + rank] = tid;
    if (rank == 0) {
      int dd = 0, gp = 0;
      for (int q = 0; q < P; ++q) {
        const int fg = first_g[q];
        if (fg > 0 && ids_s[q] < e) {
          ++dd;
          gp += fg;
        }
      }
      c.r_act[dd] = e;
      c.r_base[dd] = less;
      c.r_gpre[dd] = gp;
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
    c.r_base[n] = tot;
    c.r_gpre[n] = gt;
    *c.r_n = n;
  }
  __syncthreads();
}

// The grouping as the kernels read it: shared memory (indexed by active
// expert) or the routing kernel's output (offsets indexed by expert id).
struct Grouping {
  bool local;
  const int32_t* act;
  const int32_t* gpre;
  const int32_t* spair;
  const int32_t* r_base;
  const int32_t* offsets;
  int n_act;
  __device__ __forceinline__ int base(int d, int e) const { return local ? r_base[d] : offsets[e]; }
  __device__ __forceinline__ int end(int d, int e) const { return local ? r_base[d + 1] : offsets[e + 1]; }
};

__device__ __forceinline__ Grouping grouping_view(const GemmParams& p, const CtaSmem& c) {
  Grouping g;
  g.local = p.local != 0;
  g.act = g.local ? c.r_act : p.active;
  g.gpre = g.local ? c.r_gpre : p.gprefix;
  g.spair = g.local ? c.r_pair : p.sorted_pair;
  g.r_base = c.r_base;
  g.offsets = p.offsets;
  g.n_act = g.local ? *c.r_n : *p.n_active;
  return g;
}

// This CTA's contiguous run [u0, u1) of the work units of active experts
// [d_lo, d_hi) in one phase (unit = active expert d, 8-pair group, weight
// tile j; group-major within an expert, so a run reloads activations only at
// group boundaries; experts with more than 8 pairs stream their weights once
// per group), and the active expert d0 holding unit u0.  Every CTA gets
// floor(n / grid) units, and the n % grid remaining ones go to the CTAs of a
// window that starts at ``rot`` (wrapping); ``rot`` then moves past that
// window, so over several phases each CTA gets within one unit of its share.
struct UnitRange {
  int u0, u1, d0;
};

__device__ __forceinline__ UnitRange cta_units(const Grouping& gr, int tiles, int d_lo, int d_hi, int& rot) {
  const int G = gridDim.x, b = blockIdx.x;
  const int U0 = gr.gpre[d_lo] * tiles;
  const int n = gr.gpre[d_hi] * tiles - U0;
  const int base = n / G, rem = n - base * G;
  // CTAs c < b holding one of the rem extra units: ((c - rot) mod G) < rem
  int before;
  if (rot + rem <= G) before = min(max(b - rot, 0), rem);
  else before = min(b, rot + rem - G) + max(b - rot, 0);
  const bool extra = ((b - rot + G) % G) < rem;
  UnitRange r;
  r.u0 = U0 + b * base + before;
  r.u1 = r.u0 + base + (extra ? 1 : 0);
  rot = (rot + rem) % G;
  int lo = d_lo, hi = d_hi;  // largest d with gpre[d] * tiles <= u0
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (gr.gpre[mid] * tiles <= r.u0) lo = mid; else hi = mid;
  }
  r.d0 = lo;
  return r;
}

// The CTA whose run of a phase split with rot = 0 holds unit u (n units over
// the grid: the first n % grid CTAs get one extra).
__device__ __forceinline__ int cta_of_unit(int u, int n) {
  const int G = gridDim.x, base = n / G, rem = n - base * G;
  if (u < (base + 1) * rem) return u / (base + 1);
  return base ? rem + (u - (base + 1) * rem) / base : G - 1;
}

// Position in an mbarrier ring, carried from one phase into the next.
struct RingPos {
  int n;           // slots taken so far
  int slot;
  uint32_t parity;
  __device__ __forceinline__ void advance(int size) {
    ++n;
    if (++slot == size) {
      slot = 0;
      parity ^= 1u;
    }
  }
};

// ------------------------------------------------------------------ roles

// Producer warp: one cp.async.bulk per weight row of each unit into the next
// free stage, plus the unit's scale rows.
template <bool GATE_UP>
__device__ void produce_units(const GemmParams& p, const Grouping& gr, const UnitRange& r, const CtaSmem& c,
                              uint64_t policy, RingPos& ring) {
  const int lane = threadIdx.x & 31;
  const int S = p.n_stages, Kh = p.K >> 1;
  UnitCursor cur;
  if (r.u0 < r.u1) cur.init(gr.gpre, p.tiles, r.d0, r.u0);
  for (int u = r.u0; u < r.u1; ++u) {
    if (*c.abort_flag) return;
    if (u > r.u0) cur.next(gr.gpre, p.tiles, u);
    const int j = cur.j;
    if (ring.n >= S && !mbar_wait(&c.empty[ring.slot], ring.parity ^ 1u, p.status, p.wait_ns)) {
      *c.abort_flag = 1;
      return;
    }
    const int e = chk(gr.act[cur.d], p.E, p.status);
    uint8_t* sw = c.stages + (size_t)ring.slot * p.stage_bytes;
    uint8_t* ss = sw + kRows * p.row_stride;
    if (lane == 0) mbar_arrive_expect_tx(&c.full[ring.slot], kRows * (Kh + p.srow_bytes));
    __syncwarp();
    {
      const int row = chk(item_row<GATE_UP>(lane, j, p.I), p.N, p.status);
      bulk_g2s(sw + lane * p.row_stride, p.w + ((size_t)e * p.N + row) * Kh, Kh, &c.full[ring.slot], policy);
    }
    if (lane < (GATE_UP ? 2 : 1)) {
      // scales: gemm1 gate rows then up rows (each contiguous); gemm2 all rows
      const int rows = GATE_UP ? kRows / 2 : kRows;
      const int row0 = chk(item_row<GATE_UP>(lane * (kRows / 2), j, p.I), p.N - rows + 1, p.status);
      const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws) + ((size_t)e * p.N + row0) * p.srow_bytes;
      bulk_g2s(ss + lane * (kRows / 2) * p.srow_bytes, src, rows * p.srow_bytes, &c.full[ring.slot], policy);
    }
    ring.advance(S);
  }
}

// Before the CTA may exit: wait for the last min(fills, S) fills, walking the
// ring backwards (earlier ones were consumed).
__device__ void producer_drain(const CtaSmem& c, int S, RingPos ring, uint32_t* status, uint64_t limit_ns) {
  for (int v = 0; v < (ring.n < S ? ring.n : S); ++v) {
    if (ring.slot == 0) {
      ring.slot = S - 1;
      ring.parity ^= 1u;
    } else {
      --ring.slot;
    }
    mbar_wait(&c.full[ring.slot], ring.parity, status, limit_ns);
  }
}

// Epilogue warp: sums the consumer warps' partials of each unit (lane = one
// of 8 pair columns x 4 of the unit's rows per pass) and writes the results
// (gate_up: SiLU(h_gate) * h_up into abuf; down: per-pair rows into ybuf)
// while the consumers go on with the next units.  (Reducing only the columns
// of pairs that exist, from a column-major buffer, measured slower from 16
// tokens on: its per-column add chains run one after another.)
template <bool GATE_UP>
__device__ void reduce_units(const GemmParams& p, const Grouping& gr, const UnitRange& r, const CtaSmem& c,
                             RingPos& rr) {
  const int lane = threadIdx.x & 31;
  const int col = lane % kGroup;  // this lane's pair column in every pass
  UnitCursor cur;
  if (r.u0 < r.u1) cur.init(gr.gpre, p.tiles, r.d0, r.u0);
  int cur_e = -1, cur_grp = -1;
  int my_pair = -1;   // the pair of this lane's column (-1: none)
  float my_w = 0.f;   // its router weight (gate_up with the weight on the input)
  for (int u = r.u0; u < r.u1; ++u) {
    if (u > r.u0) cur.next(gr.gpre, p.tiles, u);
    const int d = cur.d, grp = cur.grp, j = cur.j;
    const int e = chk(gr.act[d], p.E, p.status);
    const int base = chk(gr.base(d, e), p.P + 1, p.status);
    const int npairs = chk(gr.end(d, e), p.P + 1, p.status) - base;
    if (e != cur_e || grp != cur_grp) {
      cur_e = e;
      cur_grp = grp;
      const int slot = grp * kGroup + col;
      my_pair = slot < npairs ? chk(gr.spair[chk(base + slot, p.P, p.status)], p.P, p.status) : -1;
      my_w = (GATE_UP && p.rwi && my_pair >= 0) ? p.topk_w[my_pair] : 0.f;
    }
    if (!mbar_wait(&c.red_full[rr.slot], rr.parity, p.status, p.wait_ns)) {
      *c.abort_flag = 1;
      return;
    }
    const float* rb = c.red + rr.slot * kRedFloats;
    const uint16_t* bias = p.bias ? p.bias + (size_t)e * p.N : nullptr;
    if (GATE_UP) {
      constexpr int kOut = kRows / 2;  // activated outputs per unit
#pragma unroll
      for (int q = 0; q < kOut * kGroup / 32; ++q) {
        const int row = (lane + 32 * q) / kGroup;
        float hg = 0.f, hu = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          hg += rb[w * kRows * kGroup + row * kGroup + col];
          hu += rb[w * kRows * kGroup + (row + kOut) * kGroup + col];
        }
        if (my_pair >= 0) {
          if (p.aq == kActFp8) {  // FP8 inputs: the static scale, once per output
            hg *= p.ascale;
            hu *= p.ascale;
          }
          // h = (router weight) * W13 x + b13: the weight on the input scales
          // the GEMM's output exactly as it would scale x
          if (p.rwi) {
            hg *= my_w;
            hu *= my_w;
          }
          if (bias) {
            hg += bf16_lo(bias[kOut * j + row]);
            hu += bf16_lo(bias[p.I + kOut * j + row]);
          }
          if (p.clamp > 0.f) {
            hg = fminf(fmaxf(hg, -p.clamp), p.clamp);
            hu = fminf(fmaxf(hu, -p.clamp), p.clamp);
          }
          p.dst[(size_t)chk(base + grp * kGroup + col, p.P, p.status) * p.I + chk(kOut * j + row, p.I, p.status)] =
              silu(hg) * hu;
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < kRows * kGroup / 32; ++q) {
        const int row = (lane + 32 * q) / kGroup;
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) y += rb[w * kRows * kGroup + row * kGroup + col];
        if (my_pair >= 0) {
          if (p.aq == kActFp8) y *= p.ascale;  // FP8 inputs: the static scale, once per output
          if (bias) y += bf16_lo(bias[kRows * j + row]);
          p.dst[(size_t)my_pair * p.N + chk(kRows * j + row, p.N, p.status)] = y;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.red_empty[rr.slot]);
    rr.advance(kRedBufs);
  }
}

// One consumer warp's part of one unit: its blocks [wb0, wb0 + cnt) of the
// unit's 32 weight rows (two m16n8k16 tiles) times the activation fragments,
// two blocks at a time, block scale applied to each block's fp32 partial sum.
// With FOLD the scale is multiplied by each pair column's power-of-two undo
// first, so the partial sums stay at the magnitude of the result (no float32
// overflow for large block scales with tiny, up-scaled activations).
// Four 8x8 matrices of 16-bit elements from shared memory: lane L supplies the
// row address of row L % 8 of matrix L / 8 and receives, from each matrix, the
// 4 bytes of row L / 4 at byte offset 4 (L % 4) -- for packed weight rows the
// same words the MMA fragments take.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <WeightKind KIND, int NBW, bool FOLD>
__device__ __forceinline__ void unit_mainloop(const GemmParams& p, const uint8_t* sw, const uint8_t* ss, int wb0,
                                              int cnt, int g, int t, const uint32_t (&xf)[NBW][4],
                                              const float (&inv)[2], float (&acc)[kTiles][4]) {
#pragma unroll
  for (int tl = 0; tl < kTiles; ++tl) acc[tl][0] = acc[tl][1] = acc[tl][2] = acc[tl][3] = 0.f;
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  // this lane's row address for the weight loads: matrices 0 / 1 = rows 0-7 /
  // 8-15 of the tile in block b, matrices 2 / 3 the same in block b + 1
  const int lane = threadIdx.x & 31, mat = lane >> 3;
  const uint32_t wrow = smem_u32(sw) + ((lane & 7) + 8 * (mat & 1)) * p.row_stride + (mat >> 1) * 16 + wb0 * 16;
#pragma unroll
  for (int bb = 0; bb < NBW; bb += 2) {
    if (bb < cnt) {
      const int b = wb0 + bb;
#pragma unroll
      for (int tl = 0; tl < kTiles; ++tl) {
        const int row = 16 * tl + g;
        float sc[2][2];  // [row / row+8][block b / b+1]
        load_scales2<KIND>(ss, p.srow_bytes, row, b, sc, p.status);
        float m[2][2][2];  // [row / row+8][block][column 2t / 2t+1]
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (FOLD) mul_f32x2_bcast(m[r2][h][0], m[r2][h][1], sc[r2][h], inv[0], inv[1]);
            else m[r2][h][0] = m[r2][h][1] = sc[r2][h];
          }
        uint32_t wq[2][2];  // [block b / b+1][row g / g+8]: 8 packed weights each
        ldsm_x4(wrow + 16 * tl * p.row_stride + bb * 16, wq[0][0], wq[0][1], wq[1][0], wq[1][1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
          weights_to_f16<KIND>(wq[h][0], a0, a1, a2, a3);
          weights_to_f16<KIND>(wq[h][1], c0, c1, c2, c3);
          float dd[4];
          mma_f16_16816(dd, a0, c0, a1, c1, xf[bb + h][0], xf[bb + h][1], zero);
          mma_f16_16816(dd, a2, c2, a3, c3, xf[bb + h][2], xf[bb + h][3], dd);
          fma_f32x2(acc[tl][0], acc[tl][1], m[0][h][0], m[0][h][1], dd[0], dd[1]);
          fma_f32x2(acc[tl][2], acc[tl][3], m[1][h][0], m[1][h][1], dd[2], dd[3]);
        }
      }
    }
  }
}

// Consumer warps: split K, MMA each unit's weight rows against up to 8
// activation columns held in registers, hand the partial sums to the
// epilogue warp.
template <WeightKind KIND, bool GATE_UP, int NBW, int AQ>
__device__ void consume_units(const GemmParams& p, const Grouping& gr, const UnitRange& r, const CtaSmem& c,
                              RingPos& wr, RingPos& rr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int S = p.n_stages;
  const int nb = p.K >> 5;
  // even number of blocks per warp, so blocks are processed in pairs
  const int nbw = 2 * ((nb + 2 * kConsumerWarps - 1) / (2 * kConsumerWarps));
  const int wb0 = min(nb, warp * nbw);
  const int cnt = min(nbw, nb - wb0);

  uint32_t xf[NBW][4];
  float inv[2];  // power-of-two undo for accumulator columns 2t, 2t+1
  bool fold = false;  // some column of this warp scaled: undo folded into the block scales
  int cur_e = -1, cur_grp = -1;
  int cur_tok = -2;  // gate_up: the token whose x row this lane's fragments hold (-1: none)
  UnitCursor cur;
  if (r.u0 < r.u1) cur.init(gr.gpre, p.tiles, r.d0, r.u0);
  for (int u = r.u0; u < r.u1; ++u) {
    if (*c.abort_flag) return;
    if (u > r.u0) cur.next(gr.gpre, p.tiles, u);
    const int d = cur.d, grp = cur.grp;
    const int e = chk(gr.act[d], p.E, p.status);
    const int base = chk(gr.base(d, e), p.P + 1, p.status);
    const int npairs = chk(gr.end(d, e), p.P + 1, p.status) - base;
    if (e != cur_e || grp != cur_grp) {
      // gate_up fragments are rows of x: a group with the same tokens as the
      // last one (one token: every expert's group) needs no reload.  Checked
      // only where the grouping is in shared memory (a cheap read).
      bool same = false;
      int tok = -1;
      if (GATE_UP && gr.local) {
        const int slot = grp * kGroup + g;
        if (slot < npairs) tok = chk(gr.spair[chk(base + slot, p.P, p.status)], p.P, p.status) / p.topk;
        same = __all_sync(0xffffffffu, tok == cur_tok);
      }
      if (!same) {
        load_frags<KIND, GATE_UP, NBW, AQ>(p, gr.spair, grp * kGroup, base, npairs, wb0, cnt, g, t, xf, inv);
        fold = __any_sync(0xffffffffu, inv[0] != 1.f || inv[1] != 1.f);
        cur_tok = tok;
      }
      cur_e = e;
      cur_grp = grp;
    }
    if (!mbar_wait(&c.full[wr.slot], wr.parity, p.status, p.wait_ns)) {
      *c.abort_flag = 1;
      return;
    }
    const uint8_t* sw = c.stages + (size_t)wr.slot * p.stage_bytes;
    const uint8_t* ss = sw + kRows * p.row_stride;

    // ---- main loop over this warp's 32-element blocks (fold: the
    // activations were scaled, so their undo joins the block scales)
    float acc[kTiles][4];
    if (fold) unit_mainloop<KIND, NBW, true>(p, sw, ss, wb0, cnt, g, t, xf, inv, acc);
    else unit_mainloop<KIND, NBW, false>(p, sw, ss, wb0, cnt, g, t, xf, inv, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.empty[wr.slot]);
    wr.advance(S);

    // ---- hand the partial sums to the epilogue warp
    if (rr.n >= kRedBufs && !mbar_wait(&c.red_empty[rr.slot], rr.parity ^ 1u, p.status, p.wait_ns)) {
      *c.abort_flag = 1;
      return;
    }
    // (the activations' undo is in the partial sums already: folded into the
    // block scales, or 1 when no column was scaled)
    float* rw = c.red + rr.slot * kRedFloats + warp * (kRows * kGroup);
#pragma unroll
    for (int tl = 0; tl < kTiles; ++tl) {
      const int row = 16 * tl + g;
      *reinterpret_cast<float2*>(rw + row * kGroup + 2 * t) = make_float2(acc[tl][0], acc[tl][1]);
      *reinterpret_cast<float2*>(rw + (row + 8) * kGroup + 2 * t) = make_float2(acc[tl][2], acc[tl][3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.red_full[rr.slot]);
    rr.advance(kRedBufs);
  }
}

// ------------------------------------------------------------------ kernels

// One GEMM stage (gate_up with the activation, or down) as its own launch.
template <WeightKind KIND, bool GATE_UP, int NBW, int AQ>
__global__ void __launch_bounds__(kDecThreads, 1) decode_gemm_kernel(const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const CtaSmem c = carve_smem(smem);
  const int warp = threadIdx.x >> 5;
  init_barriers(c, p.n_stages);
  // gate_up reads the grouping of the kernel before it; down reads only
  // weights and grouping here and waits for gate_up's activations further down
  if (GATE_UP) grid_dep_wait();
  grid_dep_launch_dependents();
  if (p.local) local_grouping(p, c);
  const Grouping gr = grouping_view(p, c);
  int rot = 0;
  const UnitRange r = cta_units(gr, p.tiles, 0, gr.n_act, rot);
  RingPos wr{0, 0, 0u}, rr{0, 0, 0u};
  if (warp == kProducerWarp) {
    produce_units<GATE_UP>(p, gr, r, c, l2_policy_evict_first(), wr);
    producer_drain(c, p.n_stages, wr, p.status, p.wait_ns);
    return;
  }
  if (warp == kEpilogueWarp) {
    reduce_units<GATE_UP>(p, gr, r, c, rr);
    return;
  }
  if (!GATE_UP) grid_dep_wait();  // the activations come from the gate_up kernel
  consume_units<KIND, GATE_UP, NBW, AQ>(p, gr, r, c, wr, rr);
}

// Both GEMM stages in one persistent, cooperative launch (grid = the CTAs
// that can be resident at once).  The weight stream runs on from the gate_up
// units into the down units without a gap; the down units' activations come
// from every CTA, so before its first down unit a CTA waits until all CTAs
// have published their gate_up results.  Publication: each CTA's epilogue
// warp writes the call's token into its own flag (release) after its last
// activation store; the waiting warp reads all flags (relaxed, then one
// acquire fence).  The token is epoch + 1, the epoch word being advanced by
// CTA 0 once every CTA has published (so every CTA read it before); the
// published values differ per CTA and per token, so flags left by earlier
// calls (or any constant fill) never match: the flags and the epoch need no
// clearing between calls.  (Splitting each phase into two halves of the
// experts, so the wait for the first half hides behind the second half's
// units, measured slower: every CTA then reloads its activation fragments in
// twice as many places, and each reload is a global-memory round trip of
// about 2 us under the full weight stream.)
template <WeightKind KIND, int NBW, int AQ>
__global__ void __launch_bounds__(kDecThreads, 1) decode_fused_kernel(const GemmParams p1, const GemmParams p2) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const CtaSmem c = carve_smem(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_barriers(c, p1.n_stages);
  grid_dep_wait();  // the grouping of the routing kernel; the previous call's epoch
  grid_dep_launch_dependents();
  if (threadIdx.x == 0) *c.token = ld_acquire_gpu(p1.epoch) + 1u;
  if (p1.local) local_grouping(p1, c);
  __syncthreads();
  const uint32_t token = *c.token;
  const Grouping gr = grouping_view(p1, c);
  int rot = 0;
  const UnitRange r1 = cta_units(gr, p1.tiles, 0, gr.n_act, rot);
  const UnitRange r2 = cta_units(gr, p2.tiles, 0, gr.n_act, rot);
  RingPos wr{0, 0, 0u}, rr{0, 0, 0u};
  if (warp == kProducerWarp) {
    const uint64_t policy = l2_policy_evict_first();
    produce_units<true>(p1, gr, r1, c, policy, wr);
    produce_units<false>(p2, gr, r2, c, policy, wr);
    producer_drain(c, p1.n_stages, wr, p1.status, p1.wait_ns);
    return;
  }
  if (warp == kEpilogueWarp) {
    reduce_units<true>(p1, gr, r1, c, rr);
    // publish (also after an abort, so the other CTAs do not wait it out)
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_gpu(p1.flags + blockIdx.x, published_value(token, blockIdx.x));
    reduce_units<false>(p2, gr, r2, c, rr);
    return;
  }
  consume_units<KIND, true, NBW, AQ>(p1, gr, r1, c, wr, rr);
  if (r2.u0 < r2.u1) {
    // the down units' activations come from the gate_up units of the same
    // experts: wait for the CTAs whose gate_up runs hold those units only
    if (warp == 0) {
      int d_last = r2.d0;
      while (gr.gpre[d_last + 1] * p2.tiles <= r2.u1 - 1) ++d_last;
      const int n1 = gr.gpre[gr.n_act] * p1.tiles;
      const int b_lo = cta_of_unit(gr.gpre[r2.d0] * p1.tiles, n1);
      const int b_hi = cta_of_unit(gr.gpre[d_last + 1] * p1.tiles - 1, n1);
      if (!wait_published_range(p1.flags, b_lo, b_hi + 1, token, p1.status, p1.wait_ns) && lane == 0)
        *c.abort_flag = 1;
    }
    named_bar_sync(1, kConsumerWarps * 32);
    consume_units<KIND, false, NBW, AQ>(p2, gr, r2, c, wr, rr);
  }
  // CTA 0 advances the epoch once every CTA has published (so every CTA has
  // read it); by the end of its own work that has long happened
  if (blockIdx.x == 0 && warp == 0) {
    wait_published_range(p1.flags, 0, gridDim.x + p1.wait_extra, token, p1.status, p1.wait_ns);
    if (lane == 0) *p1.epoch = token;
  }
}

__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ ybuf,
                                                      const int32_t* __restrict__ ids,
                                                      const float* __restrict__ topk_w, int E, int topk,
                                                      int H, uint16_t* __restrict__ out,
                                                      const int32_t* __restrict__ emap, int G, int rwi) {
  __shared__ int s_ids[64];
  __shared__ float s_w[64];
  // the next kernel on the stream may start its prologue now; it waits
  // (griddepcontrol.wait) for this grid to complete before using anything
  grid_dep_launch_dependents();
  // ids and router weights are read before the wait for the GEMM kernel: they
  // are inputs of the call, written before the call's first kernel, which
  // waited for all earlier work before it let this grid launch
  const int t = blockIdx.y;
  if (threadIdx.x < topk) {
    s_ids[threadIdx.x] = local_expert(ids, t * topk + threadIdx.x, emap, G, E);
    s_w[threadIdx.x] = rwi ? 1.f : topk_w[t * topk + threadIdx.x];
  }
  grid_dep_wait();  // ybuf comes from the down kernel
  __syncthreads();
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* yb = reinterpret_cast<const float4*>(ybuf + (size_t)t * topk * H) + c4;
  const int h4 = H / 4;
  // all of a round's loads are issued before any use (one memory latency per
  // 16 slots: a whole top-15 token in one round)
  for (int k0 = 0; k0 < topk; k0 += 16) {
    float4 y[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const bool valid = k0 + k < topk && (unsigned)s_ids[k0 + k] < (unsigned)E;
      y[k] = valid ? __ldcg(yb + (size_t)(k0 + k) * h4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
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

template <WeightKind KIND, bool GATE_UP, int NBW, int AQ>
cudaError_t launch_gemm(const GemmParams& gp, int grid, cudaStream_t s) {
  const size_t smem = kSmemFixed + (size_t)gp.n_stages * gp.stage_bytes;
  auto kern = decode_gemm_kernel<KIND, GATE_UP, NBW, AQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(kDecThreads), smem, s, true, false, gp);
}

// activation blocks of 32 per consumer warp (even), which sizes the register fragments
int blocks_per_warp(int K) { return 2 * (((K >> 5) + 2 * kConsumerWarps - 1) / (2 * kConsumerWarps)); }

template <WeightKind KIND, bool GATE_UP, int AQ>
cudaError_t dispatch_nbw(const GemmParams& gp, int grid, cudaStream_t s) {
  const int nbw = blocks_per_warp(gp.K);
  if (nbw <= 8) return launch_gemm<KIND, GATE_UP, 8, AQ>(gp, grid, s);
  if (nbw <= 16) return launch_gemm<KIND, GATE_UP, 16, AQ>(gp, grid, s);
  return cudaErrorInvalidValue;  // K above 7168: outside the size limits
}

// The kernel variants a call uses: int4 weights never come with quantised
// activations (the library rejects the combination).
template <bool GATE_UP>
cudaError_t dispatch_gemm(const GemmParams& gp, WeightKind kind, int grid, cudaStream_t s) {
  if (kind == WeightKind::kInt4) return dispatch_nbw<WeightKind::kInt4, GATE_UP, kActNone>(gp, grid, s);
  if (kind == WeightKind::kInt4Bf16) return dispatch_nbw<WeightKind::kInt4Bf16, GATE_UP, kActNone>(gp, grid, s);
  if (gp.aq == kActMxfp4) return dispatch_nbw<WeightKind::kMxfp4, GATE_UP, kActMxfp4>(gp, grid, s);
  if (gp.aq == kActFp8) return dispatch_nbw<WeightKind::kMxfp4, GATE_UP, kActFp8>(gp, grid, s);
  return dispatch_nbw<WeightKind::kMxfp4, GATE_UP, kActNone>(gp, grid, s);
}

// The fused kernel holds fragments for up to 8 blocks per warp (K <= 3584 in
// both GEMMs).
constexpr int kFusedNbw = 8;

// CTAs of the fused kernel that can be resident at once on this device (0 if
// the device cannot launch cooperative grids or a query fails).  Its CTAs
// wait on one another, so it is launched as a cooperative grid of this size:
// the launch then either places every CTA at once or fails, instead of
// leaving CTAs waiting for others that cannot be scheduled.
template <WeightKind KIND, int AQ>
int fused_resident_ctas(size_t smem, int sms) {
  auto kern = decode_fused_kernel<KIND, kFusedNbw, AQ>;
  int dev = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem) != cudaSuccess) return 0;
  return per_sm * sms;
}

template <WeightKind KIND, int AQ>
cudaError_t launch_fused(const GemmParams& g1, const GemmParams& g2, int grid, cudaStream_t s) {
  const size_t smem = kSmemFixed + (size_t)g1.n_stages * g1.stage_bytes;
  auto kern = decode_fused_kernel<KIND, kFusedNbw, AQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(kDecThreads), smem, s, true, true, g1, g2);
}

int stage_bytes_for(int K, WeightKind kind, int* row_stride, int* srow_bytes) {
  *row_stride = (K >> 1) + 16;
  *srow_bytes = (K >> 5) * scale_bytes(kind);
  const int raw = kRows * *row_stride + kRows * *srow_bytes;
  return (raw + 127) & ~127;
}

// Stage size and count; with ``other`` (fused kernel) one ring serves both
// GEMMs, its stages sized for the larger.
void fill_stage_geometry(GemmParams& gp, WeightKind kind, const GemmParams* other = nullptr) {
  int stage = stage_bytes_for(gp.K, kind, &gp.row_stride, &gp.srow_bytes);
  if (other) {
    int rs, sb;
    stage = max(stage, stage_bytes_for(other->K, kind, &rs, &sb));
  }
  gp.stage_bytes = stage;
  const int st = (kSmemBudget - kSmemFixed) / stage;
  gp.n_stages = st > kMaxStages ? kMaxStages : st;
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
  g1.epoch = a.sync;
  g1.flags = a.sync ? a.sync + kSyncFlagsOffset : nullptr;
  g1.wait_ns = a.wait.limit_ns;
  g1.wait_extra = 0;
  g1.topk_w = a.topk_w;
  g1.bias = a.opt.b13;
  g1.emap = a.opt.emap;
  g1.G = a.opt.G;
  g1.rwi = a.opt.rwi;
  g1.aq = a.opt.aq;
  g1.ascale = a.opt.s13;
  g1.clamp = a.opt.clamp;

  GemmParams g2 = g1;
  g2.ascale = a.opt.s2;
  g2.w = a.w2;
  g2.ws = a.w2_s;
  g2.N = a.H;
  g2.K = a.I;
  g2.tiles = a.H / kRows;
  g2.src = a.abuf;
  g2.dst = a.ybuf;
  g2.bias = a.opt.b2;

  const int aq = a.opt.aq;  // quantised activations: MXFP4 weights only (checked by the library)
  // one launch for both GEMMs when both fit the fused kernel's fragments and a
  // resident grid fits the flag array
  bool fused = a.sync != nullptr && blocks_per_warp(a.H) <= kFusedNbw && blocks_per_warp(a.I) <= kFusedNbw;
  int fused_grid = 0;
  if (fused) {
    fill_stage_geometry(g1, a.kind, &g2);
    fill_stage_geometry(g2, a.kind, &g1);
    const size_t smem = kSmemFixed + (size_t)g1.n_stages * g1.stage_bytes;
    fused_grid = a.kind == WeightKind::kInt4 ? fused_resident_ctas<WeightKind::kInt4, kActNone>(smem, a.num_sms)
                 : a.kind == WeightKind::kInt4Bf16
                     ? fused_resident_ctas<WeightKind::kInt4Bf16, kActNone>(smem, a.num_sms)
                 : aq == kActMxfp4 ? fused_resident_ctas<WeightKind::kMxfp4, kActMxfp4>(smem, a.num_sms)
                 : aq == kActFp8   ? fused_resident_ctas<WeightKind::kMxfp4, kActFp8>(smem, a.num_sms)
                                   : fused_resident_ctas<WeightKind::kMxfp4, kActNone>(smem, a.num_sms);
    g1.wait_extra = a.wait.extra_waiters;
    fused = fused_grid >= 1 && g1.n_stages >= 2 && fused_grid + a.wait.extra_waiters <= kMaxSyncCtas;
  }
  if (!fused) {
    fill_stage_geometry(g1, a.kind, nullptr);
    fill_stage_geometry(g2, a.kind, nullptr);
    g1.wait_extra = 0;
  }
  if (g1.n_stages < 2 || g2.n_stages < 2) return cudaErrorInvalidValue;

  cudaError_t e;
  if (fused) {
    timing_mark(1, false, s);
    e = a.kind == WeightKind::kInt4       ? launch_fused<WeightKind::kInt4, kActNone>(g1, g2, fused_grid, s)
        : a.kind == WeightKind::kInt4Bf16 ? launch_fused<WeightKind::kInt4Bf16, kActNone>(g1, g2, fused_grid, s)
        : aq == kActMxfp4                 ? launch_fused<WeightKind::kMxfp4, kActMxfp4>(g1, g2, fused_grid, s)
        : aq == kActFp8                   ? launch_fused<WeightKind::kMxfp4, kActFp8>(g1, g2, fused_grid, s)
                                          : launch_fused<WeightKind::kMxfp4, kActNone>(g1, g2, fused_grid, s);
    timing_mark(1, true, s);
    if (e != cudaSuccess) {
      // a cooperative grid that cannot be placed (for example under an SM
      // limit) fails at launch: outside stream capture the call goes on with
      // the two-launch path, under capture the error is returned
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return e;
      (void)cudaGetLastError();
      fused = false;
      fill_stage_geometry(g1, a.kind, nullptr);
      fill_stage_geometry(g2, a.kind, nullptr);
      g1.wait_extra = 0;
    } else {
      timing_mark(2, false, s);
      timing_mark(2, true, s);
    }
  }
  if (!fused) {
    timing_mark(1, false, s);
    e = dispatch_gemm<true>(g1, a.kind, a.num_sms, s);
    timing_mark(1, true, s);
    if (e != cudaSuccess) return e;
    timing_mark(2, false, s);
    e = dispatch_gemm<false>(g2, a.kind, a.num_sms, s);
    timing_mark(2, true, s);
    if (e != cudaSuccess) return e;
  }
  dim3 cgrid((a.H / 4 + 127) / 128, a.T);
  timing_mark(3, false, s);
  e = launch_kernel(combine_kernel, cgrid, dim3(128), 0, s, true, false, (const float*)a.ybuf, a.topk_ids, a.topk_w, a.E,
                    a.topk, a.H, reinterpret_cast<uint16_t*>(a.out), a.opt.emap, a.opt.G, a.opt.rwi);
  timing_mark(3, true, s);
  return e;
}

}  // namespace moe
