// Tensor-core grouped GEMMs for large batches (prefill): tcgen05 MMAs with the
// dequantised weights and the accumulators in tensor memory, activations by
// TMA in shared memory.
//
// Same two stages as the weight-streaming path (Mxfp4MoEMethod.apply on the
// vLLM quantization/mxfp4 API page, gate_up ``w13`` then down ``w2``), laid
// out for a dense contraction:
//   gather:  xs[i] = x[token of sorted pair i]                 (bf16 rows)
//   gemm1:   h = W13[e] xs^T, a = SiLU(h_gate) * h_up -> af    (f32)
//   convert: a16[i] = f16(af[i] * 2^aexp[i]), aexp[i] putting row i's largest
//            |a| in [2^14, 2^15)                               (f16 rows)
//   gemm2:   y = W2[e] a^T on f16 operands (weight row m scaled by 2^ew[m]),
//            outacc[t] += topk_w * y * 2^-(ew + aexp)          (fp32, red.add)
//   cast:    out = bf16(outacc)
//
// Work item = (expert, up to 192 (gate_up) or 128 (down) of its sorted rows,
// one tile of 128 weight rows; gemm1 tiles hold 64 gate rows and the matching
// 64 up rows).  The MMA is D[128 weight rows][rows] += W[128][16] X[rows][16]^T:
// M = 128 from the
// weight tile in tensor memory, N = the item's row count rounded up to 16
// from the activation tile in shared memory, so a short item costs only the
// MMA work of its own rows.
//
// Two CTAs per SM, each with its own MMA-issuing thread, take turns on the
// SM's tensor core.  A thread that issues tcgen05.mma leaves the tensor core
// idle for every cycle it spends elsewhere (a barrier wait, descriptor
// arithmetic, waiting for its epilogue to drain the accumulator); the other
// CTA's MMAs fill those gaps.  So each CTA keeps one accumulator and half of
// the SM's tensor memory and shared memory.  Items go round-robin over all
// CTAs.  Gate_up items are wider (192 rows) than down items (128) because
// every item converts its 128 x K weight tile once: more rows per item means
// fewer conversions per MMA.
//
// The pipeline runs in steps of 64 of K, 4 MMAs per step (one 64-column
// activation tile).  Shared memory holds only the activation ring (four
// gate_up or six down steps deep, enough to cover the L2 latency of the TMA
// loads); the converters read the packed weights and scales straight from
// global memory, one group of four steps ahead, into registers.
// Gate_up multiplies bf16 operands (weights exact in bf16, x bf16); down
// multiplies f16 operands: the intermediate a has 11 significant bits there
// (a bf16 a alone, 8 bits, is too coarse for the layer's tolerance) and the
// weights are exact in f16 when their block scale lies within 2^36 of the
// row's largest block scale (smaller blocks lose low bits, at 2^-37 of the
// row's largest weights).
// Warp roles per CTA:
//   warp 0      lane 0: TMA of the step's rows x 64 activation tile
//               (SWIZZLE_128B, the canonical K-major layout tcgen05 reads)
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2-9   weight converters: thread = one weight row (its TMEM lane)
//               and one of the step's two 32-element blocks; loads its 16
//               packed bytes and its scale, converts them exactly (gate_up:
//               bf16 by cvt.rn.f16x2.e2m1x2, f16 -> bf16 re-bias and the block
//               scale; down: f16 times 2^(s - 127 + ew[row])) and stores them
//               into the step's tensor-memory weight stage with tcgen05.st
//               int4_per_group_32 weights: q exact to f16 by a mantissa
//               trick, then bf16(fl32(q * s)) (gate_up) or
//               f16(q * f16(s * 2^ew[row])) (down)
//   warps 10-13 epilogue: tcgen05.ld of the accumulator, SiLU gating (gemm1)
//               or the exponent undo and router-weighted scatter-add (gemm2),
//               global stores
// Tensor memory per CTA (256 columns): two (gate_up) or four (down) 32-column
// weight stages, then one accumulator of 192 (gate_up) or 128 (down) columns.
#include <cuda.h>

#include "common.cuh"

namespace moe {

namespace {

constexpr int kConvWarps = 8;
constexpr int kEpiWarp0 = 2 + kConvWarps;
constexpr int kPThreads = (kEpiWarp0 + 4) * 32;
constexpr int kWCols = 32;                    // tensor-memory columns per weight stage (64 of K)
constexpr int kGroupSteps = 4;                // steps per converter load group (256 of K)
constexpr uint32_t kTmemCols = 256;

// Tile rows, pipeline depths, tensor-memory and shared-memory layout of one
// CTA; an activation stage holds one tile.
template <bool GATE_UP>
struct TcLayout {
  static constexpr int kRows = GATE_UP ? kTcRowsUp : kTcRowsDown;  // MMA N, at most
  static constexpr int kBoxBytes = kRows * 128;                   // one tile: kRows rows x 64 16-bit values
  static constexpr int kActStages = GATE_UP ? 4 : 6;
  static constexpr int kStageBytes = kBoxBytes;
  static constexpr int kWStages = GATE_UP ? 2 : 4;
  static constexpr uint32_t kAccCol0 = kWStages * kWCols;         // accumulator columns [kAccCol0, +kRows)
  static_assert(kAccCol0 + kRows <= kTmemCols, "tensor memory budget");
  static_assert(kRows % 32 == 0 && kRows <= 256, "MMA N limit");
  // activation ring | mbarriers; + 1024 for aligning the base: two CTAs per
  // SM need at most 113 KB each
  static constexpr int kBarOff = kActStages * kStageBytes;
  static constexpr int kEwOff = kBarOff + 256;                    // down: [2][128] weight-row exponents
  static constexpr int kSmemBytes = 1024 + kEwOff + 2 * kTcW * 4;
  static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
};

struct TcParams {
  const uint8_t* w;   // packed [E][N][K/2]
  const void* ws;     // scales [E][N][K/32]: E8M0 bytes (MXFP4) or fp32 (int4)
  int N, K, I, H;
  int n_tiles;        // weight tiles per expert
  const int32_t* mtiles;
  const int32_t* n_mtiles;
  const int32_t* offsets;
  const int32_t* counts;
  const int32_t* sorted_pair;
  int topk;
  const float* topk_w;
  float* act_out;     // gemm1: [P][I] f32, the activated intermediate
  const int32_t* aexp;  // gemm2: [P] power-of-two exponent of each f16 intermediate row
  float* outacc;      // gemm2: [T][H]
  uint32_t* status;
  uint64_t wait_ns;   // limit of every bounded wait
  const uint16_t* bias;  // bf16 [E][N] added to the outputs (gate_up: b13, down: b2), or null
  int rwi;            // router weight on the input: gate_up scales h by it, down adds unweighted
  int E, P;           // experts, pairs (T * topk): the bounds the checked build tests indices against
  float clamp;        // gate_up: outputs clamped to [-clamp, clamp] before the gating (0: off)
  float ascale;       // FP8 activations: the static scale of this GEMM's input (applied to the
                      // float32 sums; the operands hold the e4m3 values); 1 otherwise
};

// ------------------------------------------------------------------ tcgen05 / TMA helpers

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D f32, A and B both bf16 (or both f16),
// both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool bf16) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) (+)= A (tensor memory) * B (shared memory descriptor)^T,
// kind::f16 (bf16 or f16 operands, as the instruction descriptor says).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit columns of the calling thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint4 (&c)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(c[0].x), "r"(c[0].y), "r"(c[0].z), "r"(c[0].w), "r"(c[1].x), "r"(c[1].y), "r"(c[1].z), "r"(c[1].w),
      "r"(c[2].x), "r"(c[2].y), "r"(c[2].z), "r"(c[2].w), "r"(c[3].x), "r"(c[3].y), "r"(c[3].z), "r"(c[3].w)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void red_add(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Two exact E2M1 values as f16 (one packed byte) -> the same values times
// 2^-112 as bf16: the f16 exponent field and mantissa bit move down 3 bits
// into the bf16 layout, sign kept, zero stays zero.
__device__ __forceinline__ uint32_t f16pair_to_bf16_rebias(uint32_t h) {
  return ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
}

// 32 E2M1 values (16 packed bytes) of one block with E8M0 scale s -> 16 words
// of two bf16 (K order, lower element in the low half), exact.
__device__ __forceinline__ void dequant_block(const uint4& q, uint32_t s, uint4 (&out)[4]) {
  // value * 2^-112 * 2^(s-15) = value * 2^(s-127); 2^(s-15) is a normal bf16 for s <= 142
  const bool big = s > 142u;
  const uint32_t e1 = big ? 127u + 127u : s - 15u + 127u;
  const uint32_t f1 = (e1 << 7) | (e1 << 23);
  const uint32_t e2 = big ? s - 142u + 127u : 127u;
  const uint32_t f2 = (e2 << 7) | (e2 << 23);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h0, h1, h2, h3;
    e2m1x8_to_f16x8(w[i], h0, h1, h2, h3);
    uint32_t b0 = bf16x2_mul(f16pair_to_bf16_rebias(h0), f1);
    uint32_t b1 = bf16x2_mul(f16pair_to_bf16_rebias(h1), f1);
    uint32_t b2 = bf16x2_mul(f16pair_to_bf16_rebias(h2), f1);
    uint32_t b3 = bf16x2_mul(f16pair_to_bf16_rebias(h3), f1);
    if (big) {
      b0 = bf16x2_mul(b0, f2);
      b1 = bf16x2_mul(b1, f2);
      b2 = bf16x2_mul(b2, f2);
      b3 = bf16x2_mul(b3, f2);
    }
    out[i] = make_uint4(b0, b1, b2, b3);
  }
}

__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 32 int4 values (16 packed bytes, two's complement, element 2j in the low
// nibble of byte j) of one group with fp32 scale s -> 16 words of two bf16
// (K order, lower element in the low half): bf16(fl32(q * s)).  Byte j goes
// to bytes 0 and 2 of a word; masking keeps its low nibble in the low half
// and its high nibble 4 bits up in the high half, placed in the mantissa of
// f16 1024 with each nibble's top bit flipped (q + 8, offset binary; one
// logic operation with the masking, the bits being disjoint); one f16x2 FMA
// (x1, x1/16 and -1032, -72) leaves the two exact q.
__device__ __forceinline__ uint32_t int4_pair_f16(uint32_t w, int j) {
  const uint32_t v = prmt(w, 0u, 0x4040u | (uint32_t)j | ((uint32_t)j << 8));
  uint32_t m;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(m) : "r"(v), "r"(0x00F0000Fu), "r"(0x64806408u));  // (v & mask) ^ c
  return f16x2_fma(m, 0x2C003C00u, 0xD480E408u);
}

__device__ __forceinline__ void dequant_block_int4(const uint4& q, float s, uint4 (&out)[4]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t h = int4_pair_f16(w[i], j);
      float lo, hi;
      asm("{\n .reg .f16 l, u;\n mov.b32 {l, u}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, u;\n}"
          : "=f"(lo), "=f"(hi)
          : "r"(h));
      o[j] = f32x2_to_bf16x2(lo * s, hi * s);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// 2^d as two f16 (both halves), d <= 15; d below -24 (smaller than every f16)
// gives zero.
__device__ __forceinline__ uint32_t f16x2_pow2(int d) {
  uint32_t f = 0;
  if (d >= -14) f = (uint32_t)(d + 15) << 10;
  else if (d >= -24) f = 1u << (d + 24);
  return f | (f << 16);
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 32 E2M1 values of one block with E8M0 scale s -> 16 words of two f16, the
// values times 2^(s - 127 + ew): exact for s - 127 + ew >= -23 (the product of
// a 2-significant-bit E2M1 value and a power of two stays on the f16 grid down
// to its subnormals); below, rounded to the f16 grid (or zero).
__device__ __forceinline__ void dequant_block_f16(const uint4& q, uint32_t s, int ew, uint4 (&out)[4]) {
  const uint32_t f = f16x2_pow2((int)s - 127 + ew);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h0, h1, h2, h3;
    e2m1x8_to_f16x8(w[i], h0, h1, h2, h3);
    out[i] = make_uint4(f16x2_mul(h0, f), f16x2_mul(h1, f), f16x2_mul(h2, f), f16x2_mul(h3, f));
  }
}

// 32 int4 values of one group with fp32 scale s -> 16 words of two f16:
// f16(q * f16(s * 2^ew)): q is exact in f16, the scale is rounded to f16 once
// (s * 2^ew itself is exact: a power-of-two scaling inside the float32 range)
// and the product once more.
__device__ __forceinline__ void dequant_block_int4_f16(const uint4& q, float s, int ew, uint4 (&out)[4]) {
  const uint32_t sc = f32x2_to_f16x2(s * exp2_int(ew), s * exp2_int(ew));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = f16x2_mul(int4_pair_f16(w[i], j), sc);
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Exponent ew of one weight row for the f16 down GEMM: its largest weight
// times 2^ew lies below 2^15 (6 * 2^13 for E2M1, 7 * 2^(floor(log2 smax) + 12)
// for int4), clamped to [-126, 126].  ``sr`` is the row's Kb scales.
template <WeightKind KIND>
__device__ __forceinline__ int weight_row_exponent(const uint8_t* sr, int Kb) {
  if (KIND == WeightKind::kMxfp4) {
    uint32_t m = 0;
    for (int i = 0; i < Kb; i += 16) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(sr + i));
      m = __vmaxu4(m, __vmaxu4(__vmaxu4(u.x, u.y), __vmaxu4(u.z, u.w)));
    }
    m = __vmaxu4(m, m >> 16);
    m = __vmaxu4(m, m >> 8);
    return min(140 - (int)(m & 0xFFu), 126);
  } else {
    float m = 0.f;
    if (KIND == WeightKind::kInt4) {
      for (int i = 0; i < Kb; i += 4) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(sr) + i / 4);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
      }
    } else {
      for (int i = 0; i < Kb; i += 8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(sr) + i / 8);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(wd[j])), fabsf(bf16_hi(wd[j]))));
      }
    }
    if (m == 0.f) return 0;
    const int em = max((int)((__float_as_uint(m) >> 23) & 0xFFu), 1) - 127;  // floor(log2 m), subnormals as -126
    return max(min(11 - em, 126), -126);
  }
}

struct ItemInfo {
  int e, nt, row0, rows;
};

template <int kRows>
__device__ __forceinline__ ItemInfo decode_item(const TcParams& p, int item) {
  ItemInfo it;
  const int mp = item / p.n_tiles;
  it.nt = item - mp * p.n_tiles;
  const int code = p.mtiles[mp];
  it.e = chk(code >> 20, p.E, p.status);
  const int mi = code & 0xFFFFF;
  it.row0 = chk(p.offsets[it.e] + kRows * mi, p.P, p.status);
  it.rows = chk(min(kRows, p.counts[it.e] - kRows * mi) - 1, p.P - it.row0, p.status) + 1;
  return it;
}

template <WeightKind KIND, bool GATE_UP>
__global__ void __launch_bounds__(kPThreads, 2) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                               const TcParams p) {
  using Lay = TcLayout<GATE_UP>;
  constexpr int kActStages = Lay::kActStages;
  constexpr int kWStages = Lay::kWStages;
  constexpr int kRows = Lay::kRows;
  constexpr uint32_t kAccCol0 = Lay::kAccCol0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* act_ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* act_full = bars;                  // [kActStages] activation tiles landed
  uint64_t* act_empty = act_full + kActStages;  // [kActStages] their MMAs are done
  uint64_t* w_full = act_empty + kActStages;  // [kWStages] weight stage stored by all converters
  uint64_t* w_empty = w_full + kWStages;      // [kWStages] its MMAs are done
  uint64_t* acc_full = w_empty + kWStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* ew_full = drain + 1;              // [2] down: an item's weight-row exponents written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ew_full + 2);
  int32_t* ew_s = reinterpret_cast<int32_t*>(smem + Lay::kEwOff);  // [2][kTcW]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kActStages; ++s) {
      mbar_init(&act_full[s], 1);
      mbar_init(&act_empty[s], 1);
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&w_full[s], kConvWarps);
      mbar_init(&w_empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    mbar_init(&ew_full[0], 4);
    mbar_init(&ew_full[1], 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int n_items = *p.n_mtiles * p.n_tiles;
  // a step is 64 of K: one 64-column tile of x (gate_up) or of the f16 intermediate (down)
  const int n_steps = p.K / 64;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ activation TMA
      uint32_t stage = 0, phase = 0, used = 0;
      bool stop = false;
      ItemInfo nxt{};
      if ((int)blockIdx.x < n_items) nxt = decode_item<kRows>(p, blockIdx.x);
      for (int item = blockIdx.x; item < n_items && !*abort_flag && !stop; item += gridDim.x) {
        const ItemInfo it = nxt;  // this item's routing fields were loaded an item ahead
        if (item + (int)gridDim.x < n_items) nxt = decode_item<kRows>(p, item + gridDim.x);
        for (int step = 0; step < n_steps; ++step) {
          if (used >= (uint32_t)kActStages && !mbar_wait(&act_empty[stage], phase ^ 1u, p.status, p.wait_ns)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* st = act_ring + stage * Lay::kStageBytes;
          mbar_arrive_expect_tx(&act_full[stage], Lay::kStageBytes);
          tma_load_2d(st, &tmap_a, 64 * step, it.row0, &act_full[stage]);
          ++used;
          if (++stage == (uint32_t)kActStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // nothing issued may still be in flight when the CTA exits: wait for the
      // last min(used, kActStages) stages to land
      for (uint32_t v = 0; v < (used < (uint32_t)kActStages ? used : (uint32_t)kActStages); ++v) {
        stage = stage == 0 ? kActStages - 1 : stage - 1;
        if (stage == (uint32_t)kActStages - 1) phase ^= 1u;
        mbar_wait(&act_full[stage], phase, p.status, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t as = 0, aph = 0, ws = 0, wph = 0, j = 0;
      int item = blockIdx.x;
      ItemInfo it{};
      if (item < n_items) it = decode_item<kRows>(p, item);
      const uint32_t act0 = smem_u32(act_ring);
      const uint32_t d = tmem_base + kAccCol0;
      for (; item < n_items && !*abort_flag; item += gridDim.x, ++j) {
        // the next item's routing fields, loaded a whole item ahead
        const ItemInfo nxt = item + (int)gridDim.x < n_items ? decode_item<kRows>(p, item + gridDim.x) : it;
        const uint32_t idesc = idesc_f16kind(kTcW, (it.rows + 15) & ~15, GATE_UP);  // N: the rows rounded up to 16
        // the epilogue must have read the previous item's accumulator
        if (j >= 1 && !mbar_wait(acc_empty, (j - 1) & 1u, p.status, p.wait_ns)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int step = 0; step < n_steps; ++step) {
          if (!mbar_try_wait2(&w_full[ws], wph, &act_full[as], aph) &&
              (!mbar_wait(&w_full[ws], wph, p.status, p.wait_ns) || !mbar_wait(&act_full[as], aph, p.status, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = tmem_base + ws * kWCols;
          const uint64_t b0 = sw128_desc(act0 + as * Lay::kStageBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_bf16_ta(d, a + 8 * k, b0 + 2 * k, idesc, (step > 0 || k > 0) ? 1u : 0u);
          mma_commit(&act_empty[as]);
          mma_commit(&w_empty[ws]);
          if (++as == (uint32_t)kActStages) {
            as = 0;
            aph ^= 1u;
          }
          if (++ws == (uint32_t)kWStages) {
            ws = 0;
            wph ^= 1u;
          }
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        mma_commit(acc_full);
        it = nxt;
      }
      // all issued MMAs complete before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, p.status, p.wait_ns);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------------ weight converters
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int hk = (warp - 2) >> 2;          // which of the step's two blocks
    const int L = 32 * q + lane;             // TMEM lane = weight row of the tile
    const int Kb = p.K >> 5, Kh = p.K >> 1;
    const uint32_t tl = tmem_base + ((uint32_t)(32 * q) << 16) + 16 * hk;
    // weight row of TMEM lane L within a tile: for gate_up, every 32-lane
    // quadrant holds 16 gate rows (lanes 0-15) and their 16 up rows (lanes
    // 16-31), so one epilogue warp sees both halves of its 16 activations
    const int lrow = GATE_UP ? ((L & 31) < 16 ? 16 * q + (L & 31) : p.I + 16 * q + (L & 31) - 16) : L;
    const int n_groups = n_steps / kGroupSteps;
    uint32_t ws = 0, wph = 0, used = 0;
    bool stop = false;
    // weight and scale rows of this thread for an item
    constexpr int kSB = scale_bytes(KIND);  // bytes per scale
    auto rows_of = [&](const ItemInfo& it, const uint8_t*& wr, const uint8_t*& sr) {
      const size_t row = (size_t)it.e * p.N + (GATE_UP ? 64 * it.nt : kTcW * it.nt) + lrow;
      wr = p.w + row * Kh + 16 * hk;  // block 2 * step + hk at + 32 * step
      sr = reinterpret_cast<const uint8_t*>(p.ws) + row * Kb * kSB;
    };
    // scales of one load group: MXFP4 the group's 8 E8M0 bytes; int4 this
    // thread's 4 scales (blocks hk, 2 + hk, 4 + hk, 6 + hk of the group), fp32
    // or bf16
    auto load_scales = [&](const uint8_t* sr, int g, uint2& e8, float (&f4)[4]) {
      if (KIND == WeightKind::kMxfp4) {
        e8 = __ldg(reinterpret_cast<const uint2*>(sr + 8 * g));
        chk_e8m0(e8.x, 4, p.status);
        chk_e8m0(e8.y, 4, p.status);
      } else if (KIND == WeightKind::kInt4) {
        // the group's 8 fp32 scales in two 16-byte loads (four scalar loads
        // of this thread's scales: the int4 prefill layer 5.69 ms, not 5.13)
        const float4* sf = reinterpret_cast<const float4*>(sr) + 2 * g;
        const float4 a = __ldg(sf), b = __ldg(sf + 1);
        f4[0] = hk ? a.y : a.x;
        f4[1] = hk ? a.w : a.z;
        f4[2] = hk ? b.y : b.x;
        f4[3] = hk ? b.w : b.z;
      } else {
        // the group's 8 bf16 scales in one 16-byte load; this thread's are
        // the halves hk of each word
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(sr) + g);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) f4[i] = hk ? bf16_hi(wd[i]) : bf16_lo(wd[i]);
      }
    };
    // one group = 4 steps = 8 blocks of the row: 4 blocks of this thread, 8
    // scale bytes.  qb[i] holds the block of step i of the current group and
    // is reloaded with the next group's -- the next item's first group at the
    // end of an item -- as soon as it is converted.
    uint4 qb[kGroupSteps];
    uint2 ns = make_uint2(0u, 0u);
    float nf[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t *wrow = nullptr, *srow = nullptr;
    if ((int)blockIdx.x < n_items) {
      rows_of(decode_item<kRows>(p, blockIdx.x), wrow, srow);
#pragma unroll
      for (int i = 0; i < kGroupSteps; ++i) qb[i] = __ldg(reinterpret_cast<const uint4*>(wrow + 32 * i));
      load_scales(srow, 0, ns, nf);
    }
    uint32_t jj = 0;  // items of this CTA so far
    for (int item = blockIdx.x; item < n_items && !*abort_flag && !stop; item += gridDim.x, ++jj) {
      // down: this row's f16 exponent, handed to the epilogue thread of the
      // same row (slot jj & 1: by the time an item two later is converted, the
      // epilogue has finished this one, whose accumulator the MMAs of the item
      // in between had to wait for)
      const int ew = GATE_UP ? 0 : weight_row_exponent<KIND>(srow, Kb);
      if (!GATE_UP && hk == 0) {
        ew_s[(jj & 1u) * kTcW + L] = ew;
        __syncwarp();
        if (lane == 0) mbar_arrive(&ew_full[jj & 1u]);
      }
      // the following item's rows, for the loads issued during our last group
      const bool has_next = item + (int)gridDim.x < n_items;
      const uint8_t *wrow_n = wrow, *srow_n = srow;
      if (has_next) rows_of(decode_item<kRows>(p, item + gridDim.x), wrow_n, srow_n);
      for (int g = 0; g < n_groups && !stop; ++g) {
        const uint2 cs = ns;
        float cf[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cf[i] = nf[i];
        const bool last = g + 1 == n_groups;
        const bool more = !last || has_next;
        const uint8_t* wnext = last ? wrow_n : wrow + 128 * (g + 1);
        if (more) load_scales(last ? srow_n : srow, last ? 0 : g + 1, ns, nf);
#pragma unroll
        for (int i = 0; i < kGroupSteps; ++i) {
          const int c = 2 * i + hk;  // block of the group
          uint4 cv[4];
          if (KIND == WeightKind::kMxfp4) {
            const uint32_t s = ((i < 2 ? cs.x >> (8 * c) : cs.y >> (8 * (c - 4))) & 0xFFu);
            if (GATE_UP) dequant_block(qb[i], s, cv);
            else dequant_block_f16(qb[i], s, ew, cv);
          } else {
            if (GATE_UP) dequant_block_int4(qb[i], cf[i], cv);
            else dequant_block_int4_f16(qb[i], cf[i], ew, cv);
          }
          if (more) qb[i] = __ldg(reinterpret_cast<const uint4*>(wnext + 32 * i));
          if (used >= (uint32_t)kWStages && !mbar_wait(&w_empty[ws], wph ^ 1u, p.status, p.wait_ns)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          tmem_st16(tl + ws * kWCols, cv);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&w_full[ws]);
          ++used;
          if (++ws == (uint32_t)kWStages) {
            ws = 0;
            wph ^= 1u;
          }
        }
      }
      wrow = wrow_n;
      srow = srow_n;
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    uint32_t j = 0;
    for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x, ++j) {
      const ItemInfo it = decode_item<Lay::kRows>(p, item);
      // token, router weight and (down) intermediate exponent of rows lane,
      // lane + 32, ... (loaded before the accumulator wait, handed out with
      // shuffles below): down always, gate_up for the router weight on the input
      int tok[kRows / 32], aex[kRows / 32];
      float wgt[kRows / 32];
      if (!GATE_UP || p.rwi) {
#pragma unroll
        for (int c = 0; c < kRows / 32; ++c) {
          tok[c] = 0;
          aex[c] = 0;
          wgt[c] = 0.f;
          if (32 * c + lane < it.rows) {
            const int pair = chk(p.sorted_pair[it.row0 + 32 * c + lane], p.P, p.status);
            tok[c] = pair / p.topk;
            wgt[c] = (GATE_UP || !p.rwi) ? p.topk_w[pair] : 1.f;
            if (!GATE_UP) aex[c] = p.aexp[it.row0 + 32 * c + lane];
          }
        }
      }
      // down: the f16 exponent of this thread's weight row, from its converter
      int ewr = 0;
      if (!GATE_UP) {
        if (!mbar_wait(&ew_full[j & 1u], (j >> 1) & 1u, p.status, p.wait_ns)) {
          *abort_flag = 1;
          break;
        }
        ewr = ew_s[(j & 1u) * kTcW + 32 * q + lane];
      }
      // this lane's bias: gate_up the gate and up bias of its activation
      // column, down the bias of its output row
      float bias0 = 0.f, bias1 = 0.f;
      if (p.bias) {
        const uint16_t* b = p.bias + (size_t)it.e * p.N;
        if (GATE_UP) {
          const int j1 = 64 * it.nt + 16 * q + (lane & 15);
          bias0 = bf16_lo(b[j1]);
          bias1 = bf16_lo(b[p.I + j1]);
        } else {
          bias0 = bf16_lo(b[kTcW * it.nt + 32 * q + lane]);
        }
      }
      if (!mbar_wait(acc_full, j & 1u, p.status, p.wait_ns)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + kAccCol0;
#pragma unroll
      for (int c = 0; c < kRows / 32; ++c) {
        const int c0 = 32 * c;
        if (c0 >= it.rows) break;
        uint32_t v[32];
        tmem_ld32(tbase + c0, v);
        tmem_ld_wait();
        if (GATE_UP) {
          // lanes 0-15: gate rows of activations 16q + lane, tokens c0..c0+15;
          // lanes 16-31: the matching up rows, tokens c0+16..c0+31
          const bool lo_half = lane < 16;
          float* dst = p.act_out + (size_t)(it.row0 + c0 + (lo_half ? 0 : 16)) * p.I + 64 * it.nt + 16 * q + (lane & 15);
          const int nvalid = it.rows - c0 - (lo_half ? 0 : 16);
          // exchange in place: afterwards v[i] is the gate and v[16 + i] the up
          // value of this lane's token i (all shuffles first, then independent math)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, lo_half ? v[16 + i] : v[i], 16);
            if (lo_half) v[16 + i] = recv;
            else v[i] = recv;
          }
          const size_t rs = (size_t)p.I;
          // all 16 values first, then the stores (predicated only in a partial chunk)
          float av[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float hg = __uint_as_float(v[i]) * p.ascale, hu = __uint_as_float(v[16 + i]) * p.ascale;
            if (p.rwi) {
              const float wt = __shfl_sync(0xffffffffu, wgt[c], (lo_half ? 0 : 16) + i);
              hg *= wt;
              hu *= wt;
            }
            hg += bias0;
            hu += bias1;
            if (p.clamp > 0.f) {
              hg = fminf(fmaxf(hg, -p.clamp), p.clamp);
              hu = fminf(fmaxf(hu, -p.clamp), p.clamp);
            }
            av[i] = silu(hg) * hu;
          }
          if (nvalid >= 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[i * rs] = av[i];
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i < nvalid) dst[i * rs] = av[i];
          }
        } else {
          float* dst = p.outacc + kTcW * it.nt + 32 * q + lane;
          const int nvalid = min(32, it.rows - c0);
          // y = acc * 2^-(ew + aexp) in two power-of-two steps (each exponent
          // within [-126, 126], the intermediate between acc and y)
          auto undo = [&](float acc, int ea) {
            const int k = ewr + ea, k1 = k >> 1;
            return acc * exp2_int(-k1) * exp2_int(k1 - k) * p.ascale;
          };
          if (nvalid == 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int t = __shfl_sync(0xffffffffu, tok[c], i);
              const float wk = __shfl_sync(0xffffffffu, wgt[c], i);
              const int ea = __shfl_sync(0xffffffffu, aex[c], i);
              red_add(dst + (size_t)t * p.H, wk * (undo(__uint_as_float(v[i]), ea) + bias0));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int t = __shfl_sync(0xffffffffu, tok[c], i);
              const float wk = __shfl_sync(0xffffffffu, wgt[c], i);
              const int ea = __shfl_sync(0xffffffffu, aex[c], i);
              if (i < nvalid) red_add(dst + (size_t)t * p.H, wk * (undo(__uint_as_float(v[i]), ea) + bias0));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// xs[i] = x[token of sorted pair i]: one warp per row (H <= 4096: at most 16
// sixteen-byte chunks per lane, all loads issued before the stores), eight
// rows per CTA.  With quantised activations (aq) the row is stored
// quantised-dequantised: MXFP4 code * 2^(s-127), or the FP8 e4m3 value; both
// exact in bf16.  A 32-value block is the chunks of lanes 4m .. 4m+3.
constexpr int kGatherRowsPerCta = 8;

__device__ __forceinline__ uint4 act_quant_bf16x8(uint4 u, int aq, float s) {
  float v[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
  act_quant8(aq, s, v);
  return make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]), f32x2_to_bf16x2(v[4], v[5]),
                    f32x2_to_bf16x2(v[6], v[7]));
}

__global__ void __launch_bounds__(32 * kGatherRowsPerCta) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                                            const int32_t* __restrict__ sorted_pair,
                                                                            const int32_t* __restrict__ n_valid,
                                                                            int topk, int H, int aq, float s,
                                                                            uint16_t* __restrict__ xs, int P,
                                                                            uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kGatherRowsPerCta + (threadIdx.x >> 5);
  if (i >= *n_valid) return;  // whole warps leave: the row index is per warp
  const int tok = chk(sorted_pair[chk(i, P, status)], P, status) / topk;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)tok * H);
  uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)i * H);
  const int n16 = H / 8;  // sixteen-byte chunks per row
  uint4 v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k)
    if (lane + 32 * k < n16) v[k] = __ldg(src + lane + 32 * k);
  if (aq != kActNone) {
    // chunks beyond the row are whole blocks (H % 32 == 0) of zeros
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (32 * k >= n16) break;  // warp-uniform
      if (lane + 32 * k >= n16) v[k] = make_uint4(0u, 0u, 0u, 0u);
      v[k] = act_quant_bf16x8(v[k], aq, s);
    }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k)
    if (lane + 32 * k < n16) dst[lane + 32 * k] = v[k];
}

// Row i of the activated intermediate (f32) -> f16, scaled by 2^aexp[i] so
// that the row's largest magnitude lies in [2^14, 2^15): every value within
// 2^28 of it keeps 11 significant bits.  aexp is clamped to [-126, 126]; an
// all-zero row gets 0.  One CTA of 256 threads per row, I <= 4096, 8 values
// per thread and chunk.  With quantised activations the row is quantised
// first (MXFP4 blocks of 32 = the chunks of lanes 4m .. 4m+3; the maximum is
// taken over the dequantised values); FP8 rows keep their e4m3 values (exact
// in f16) with aexp 0.
__global__ void __launch_bounds__(256) act_to_f16_kernel(const float* __restrict__ af,
                                                         const int32_t* __restrict__ n_valid, int I, int aq, float s,
                                                         uint16_t* __restrict__ a16, int32_t* __restrict__ aexp) {
  __shared__ float s_max[8];
  const int row = blockIdx.x;
  if (row >= *n_valid) return;
  const float4* src = reinterpret_cast<const float4*>(af + (size_t)row * I);
  const int n8 = I / 8;
  float v[2][8];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = threadIdx.x + 256 * i;
    const float4 a = c < n8 ? __ldcs(src + 2 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 b = c < n8 ? __ldcs(src + 2 * c + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    v[i][0] = a.x; v[i][1] = a.y; v[i][2] = a.z; v[i][3] = a.w;
    v[i][4] = b.x; v[i][5] = b.y; v[i][6] = b.z; v[i][7] = b.w;
    if (aq != kActNone) act_quant8(aq, s, v[i]);  // block-uniform: every lane calls it
#pragma unroll
    for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(v[i][q]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  m = s_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, s_max[w]);
  // floor(log2 m) from the exponent field (subnormal m counts as 2^-127)
  const int lg = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  const int ea = (m > 0.f && aq != kActFp8) ? max(min(14 - lg, 126), -126) : 0;
  const float sc = exp2_int(ea);
  uint4* dst = reinterpret_cast<uint4*>(a16 + (size_t)row * I);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = threadIdx.x + 256 * i;
    if (c < n8)
      dst[c] = make_uint4(f32x2_to_f16x2(v[i][0] * sc, v[i][1] * sc), f32x2_to_f16x2(v[i][2] * sc, v[i][3] * sc),
                          f32x2_to_f16x2(v[i][4] * sc, v[i][5] * sc), f32x2_to_f16x2(v[i][6] * sc, v[i][7] * sc));
  }
  if (threadIdx.x == 0) aexp[row] = ea;
}

__global__ void __launch_bounds__(256) cast_out_kernel(const float* __restrict__ acc, long long n4,
                                                       uint16_t* __restrict__ out) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(acc) + i);
    uint2 o;
    o.x = f32x2_to_bf16x2(v.x, v.y);
    o.y = f32x2_to_bf16x2(v.z, v.w);
    reinterpret_cast<uint2*>(out)[i] = o;
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t get_encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  if (!cached) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr) return e != cudaSuccess ? e : cudaErrorNotSupported;
    cached = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  *fn = cached;
  return cudaSuccess;
}

// 16-bit [rows][K] row-major (bf16 or f16), box_rows x 64 boxes with 128-byte swizzle.
cudaError_t make_act_map(CUtensorMap* m, const void* base, long long rows, int K, int box_rows, bool f16) {
  EncodeTiledFn enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <WeightKind KIND, bool GATE_UP>
cudaError_t launch_tc(const CUtensorMap& map, const TcParams& p, int grid, cudaStream_t s) {
  const size_t smem = (size_t)TcLayout<GATE_UP>::kSmemBytes;
  auto kern = tc_gemm_kernel<KIND, GATE_UP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kPThreads, smem, s>>>(map, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  const long long P = (long long)a.T * a.topk;
  CUtensorMap map_x, map_a;
  cudaError_t e = make_act_map(&map_x, a.xs, P, a.H, kTcRowsUp, false);
  if (e != cudaSuccess) return e;
  e = make_act_map(&map_a, a.a16, P, a.I, kTcRowsDown, true);
  if (e != cudaSuccess) return e;

  timing_mark(1, false, s);
  gather_rows_kernel<<<(unsigned)((P + kGatherRowsPerCta - 1) / kGatherRowsPerCta), 32 * kGatherRowsPerCta, 0, s>>>(
      reinterpret_cast<const uint16_t*>(a.x), a.route.sorted_pair, a.route.offsets + a.E, a.topk, a.H, a.opt.aq,
      a.opt.s13, reinterpret_cast<uint16_t*>(a.xs), (int)P, a.status);
  timing_mark(1, true, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  TcParams p{};
  p.w = a.w13;
  p.ws = a.w13_s;
  p.N = 2 * a.I;
  p.K = a.H;
  p.I = a.I;
  p.H = a.H;
  p.n_tiles = a.I / 64;
  p.mtiles = a.route.mtiles;
  p.n_mtiles = a.route.n_mtiles;
  p.offsets = a.route.offsets;
  p.counts = a.route.counts;
  p.sorted_pair = a.route.sorted_pair;
  p.topk = a.topk;
  p.topk_w = a.topk_w;
  p.act_out = a.af;
  p.aexp = a.aexp;
  p.outacc = a.outacc;
  p.status = a.status;
  p.wait_ns = a.wait_ns;
  p.bias = a.opt.b13;
  p.rwi = a.opt.rwi;
  p.ascale = a.opt.aq == kActFp8 ? a.opt.s13 : 1.f;
  p.E = a.E;
  p.P = (int)P;
  p.clamp = a.opt.clamp;
  timing_mark(2, false, s);
  e = a.kind == WeightKind::kMxfp4  ? launch_tc<WeightKind::kMxfp4, true>(map_x, p, 2 * a.num_sms, s)
      : a.kind == WeightKind::kInt4 ? launch_tc<WeightKind::kInt4, true>(map_x, p, 2 * a.num_sms, s)
                                    : launch_tc<WeightKind::kInt4Bf16, true>(map_x, p, 2 * a.num_sms, s);
  timing_mark(2, true, s);
  if (e != cudaSuccess) return e;

  timing_mark(3, false, s);
  act_to_f16_kernel<<<(unsigned)P, 256, 0, s>>>(a.af, a.route.offsets + a.E, a.I, a.opt.aq, a.opt.s2,
                                                 reinterpret_cast<uint16_t*>(a.a16), a.aexp);
  timing_mark(3, true, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if ((e = cudaMemsetAsync(a.outacc, 0, (size_t)a.T * a.H * sizeof(float), s)) != cudaSuccess) return e;
  TcParams p2 = p;
  p2.w = a.w2;
  p2.ws = a.w2_s;
  p2.N = a.H;
  p2.K = a.I;
  p2.n_tiles = a.H / kTcW;
  p2.mtiles = a.route.mtiles_dn;
  p2.n_mtiles = a.route.n_mtiles_dn;
  p2.bias = a.opt.b2;
  p2.ascale = a.opt.aq == kActFp8 ? a.opt.s2 : 1.f;
  timing_mark(4, false, s);
  e = a.kind == WeightKind::kMxfp4  ? launch_tc<WeightKind::kMxfp4, false>(map_a, p2, 2 * a.num_sms, s)
      : a.kind == WeightKind::kInt4 ? launch_tc<WeightKind::kInt4, false>(map_a, p2, 2 * a.num_sms, s)
                                    : launch_tc<WeightKind::kInt4Bf16, false>(map_a, p2, 2 * a.num_sms, s);
  timing_mark(4, true, s);
  if (e != cudaSuccess) return e;

  const long long n4 = (long long)a.T * a.H / 4;
  const int grid = (int)((n4 + 255) / 256 < (long long)a.num_sms * 8 ? (n4 + 255) / 256 : (long long)a.num_sms * 8);
  timing_mark(5, false, s);
  cast_out_kernel<<<grid, 256, 0, s>>>(a.outacc, n4, reinterpret_cast<uint16_t*>(a.out));
  timing_mark(5, true, s);
  return cudaGetLastError();
}

}  // namespace moe
