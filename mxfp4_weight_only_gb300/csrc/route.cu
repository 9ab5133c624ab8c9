// Token -> expert grouping: a stable counting sort of the T*topk (token, slot)
// pairs by expert id, in one CTA.
//
// The fused MoE call of Mxfp4MoEMethod.apply (vLLM quantization/mxfp4 API page)
// receives topk_ids[T, topk]; the grouped GEMMs need each expert's pairs
// contiguous.  Pairs keep ascending flat index p = t*topk + k inside each
// expert, ids outside [0, E) are dropped (with an expert map, global ids are
// first mapped to local ids, -1 for experts of other GPUs).  Besides counts/offsets/order this
// kernel emits the list of active experts with their 8-pair group counts
// (the weight-streaming kernels iterate over it) and, on request, the list of
// 256-row M tiles per expert for the tensor-core kernels.
#include "common.cuh"

namespace moe {

namespace {

// Exclusive scan of one value per thread over a 1024-thread CTA.
// ``scratch`` holds 32 ints.  Returns the exclusive prefix; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = scratch[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += y;
    }
    scratch[lane] = si - s;  // exclusive prefix of warp sums
    if (lane == 31) scratch[32] = si;
  }
  __syncthreads();
  const int r = incl - v + scratch[warp];
  *total = scratch[32];
  __syncthreads();
  return r;
}

// From v = the number of pairs of expert ``tid`` (0 for tid >= E) of the
// whole batch: counts, offsets, the active-expert list with its 8-pair group
// prefix and, with ``make_mtiles``, the row-tile lists of the tensor-core
// GEMMs.  Whole CTA (every thread calls it); returns this thread's offset and
// sets *total to the number of valid pairs.
__device__ int write_lists(int v, int E, int P, const RouteOut& r, int make_mtiles, int* scratch, int* total) {
  const int tid = threadIdx.x;
  const int ng = (v + kMoeGroup - 1) / kMoeGroup;
  int excl, apos, gpos, n_act, n_groups;
  if (P < 1024) {
    // counts < 2^11, active flags < 2^11, groups < 2^10: one packed scan
    int tot = 0;
    const int packed = block_excl_scan(v | ((v > 0 ? 1 : 0) << 11) | (ng << 22), scratch, &tot);
    excl = packed & 0x7FF;
    apos = (packed >> 11) & 0x7FF;
    gpos = (packed >> 22) & 0x3FF;
    *total = tot & 0x7FF;
    n_act = (tot >> 11) & 0x7FF;
    n_groups = (tot >> 22) & 0x3FF;
  } else {
    excl = block_excl_scan(v, scratch, total);
    apos = block_excl_scan(v > 0 ? 1 : 0, scratch, &n_act);
    gpos = block_excl_scan(ng, scratch, &n_groups);
  }
  if (tid < E) {
    r.counts[tid] = v;
    r.offsets[tid] = excl;
  }
  if (tid == 0) r.offsets[E] = *total;
  if (r.active) {
    if (tid < E && v > 0) {
      r.active[apos] = tid;
      r.gprefix[apos] = gpos;  // activation groups per active expert, in active-list order
    }
    if (tid == 0) {
      *r.n_active = n_act;
      r.gprefix[n_act] = n_groups;
    }
  }
  if (make_mtiles) {
    // row tiles of each expert for the two tensor-core GEMMs (counts < 2^16
    // per list here: one packed scan serves both)
    const int nt = (v + kTcRowsUp - 1) / kTcRowsUp;
    const int nd = (v + kTcRowsDown - 1) / kTcRowsDown;
    int tot = 0;
    if (P < (1 << 16)) {
      const int packed = block_excl_scan(nt | (nd << 16), scratch, &tot);
      for (int i = 0; i < nt; ++i) r.mtiles[(packed & 0xFFFF) + i] = (tid << 20) | i;
      for (int i = 0; i < nd; ++i) r.mtiles_dn[(packed >> 16) + i] = (tid << 20) | i;
      if (tid == 0) {
        *r.n_mtiles = tot & 0xFFFF;
        *r.n_mtiles_dn = tot >> 16;
      }
    } else {
      const int tpos = block_excl_scan(nt, scratch, &tot);
      for (int i = 0; i < nt; ++i) r.mtiles[tpos + i] = (tid << 20) | i;
      if (tid == 0) *r.n_mtiles = tot;
      const int dpos = block_excl_scan(nd, scratch, &tot);
      for (int i = 0; i < nd; ++i) r.mtiles_dn[dpos + i] = (tid << 20) | i;
      if (tid == 0) *r.n_mtiles_dn = tot;
    }
  }
  return excl;
}

// Stable rank of pair ``p`` (expert e, -1 if none) among the pairs of the
// same expert in this CTA's chunk of 1024 pairs, and the per-expert counts of
// the chunk in wcnt (which then holds, per warp and expert, the pairs of
// earlier warps).  ``run`` gets the chunk's count for expert tid (tid < E).
// Whole CTA; wcnt [32][E] is zeroed here.
__device__ int chunk_rank(int e, int E, int32_t* wcnt, int* run_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 32 * E; i += kRouteThreads) wcnt[i] = 0;
  __syncthreads();
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  int run = 0;
  if (tid < E) {
    for (int w = 0; w < 32; ++w) {
      const int t = wcnt[w * E + tid];
      wcnt[w * E + tid] = run;
      run += t;
    }
  }
  *run_out = run;
  __syncthreads();
  return e >= 0 ? wcnt[warp * E + e] + rank : -1;
}

// One CTA sorts every pair (batches of at most 1024 pairs, and above 2^20).
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const int32_t* __restrict__ ids, int E, int T, int topk, const int32_t* __restrict__ emap, int G,
                 RouteOut r, int make_mtiles) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;           // [E]
  int32_t* base = sm + E;      // [E]
  int32_t* wcnt = sm + 2 * E;  // [32][E]
  __shared__ int scratch[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = T * topk;

  for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0;
  // one pair per thread stays in a register when P fits one pass
  const int my_e = tid < P ? local_expert(ids, tid, emap, G, E) : -1;
  __syncthreads();
  if (P <= kRouteThreads) {
    if (my_e >= 0) atomicAdd(&cnt[my_e], 1);
  } else {
    for (int p = tid; p < P; p += kRouteThreads) {
      const int e = local_expert(ids, p, emap, G, E);
      if (e >= 0) atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();

  int n_valid = 0;
  const int excl = write_lists(tid < E ? cnt[tid] : 0, E, P, r, make_mtiles, scratch, &n_valid);
  if (tid < E) base[tid] = excl;
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  if (P <= 32) {
    // one warp holds every pair: its rank among equal ids is the position in the group
    if (warp == 0) {
      const bool valid = tid < P && (unsigned)my_e < (unsigned)E;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? my_e : -1);
      const int rank = __popc(peers & lt_mask);
      if (valid) {
        const int pos = chk(base[my_e] + rank, P, r.status);
        r.sorted_pair[pos] = tid;
        r.pair_pos[tid] = pos;
      } else if (tid < P) {
        r.pair_pos[tid] = -1;
      }
    }
  } else {
    for (int c0 = 0; c0 < P; c0 += kRouteThreads) {
      const int p = c0 + tid;
      const int e = p < P ? (c0 == 0 ? my_e : local_expert(ids, p, emap, G, E)) : -1;
      int run = 0;
      const int rank = chunk_rank(e, E, wcnt, &run);
      if (e >= 0) {
        const int pos = chk(base[e] + rank, P, r.status);
        r.sorted_pair[pos] = p;
        r.pair_pos[p] = pos;
      } else if (p < P) {
        r.pair_pos[p] = -1;
      }
      __syncthreads();
      if (tid < E) base[tid] += run;
    }
  }
  for (int i = n_valid + tid; i < P; i += kRouteThreads) r.sorted_pair[i] = -1;
}

// Large batches, step 1 of 2 (one CTA per chunk of 1024 pairs): the chunk's
// per-expert counts (hist[chunk][e]) and each pair's stable rank among the
// chunk's pairs of its expert (rank[p], -1 without an expert).
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_hist_kernel(const int32_t* __restrict__ ids, int E, int P, const int32_t* __restrict__ emap, int G,
                      int32_t* __restrict__ hist, int32_t* __restrict__ rank) {
  extern __shared__ int32_t wcnt[];  // [32][E]
  const int p = blockIdx.x * kRouteThreads + threadIdx.x;
  const int e = p < P ? local_expert(ids, p, emap, G, E) : -1;
  int run = 0;
  const int rk = chunk_rank(e, E, wcnt, &run);
  if ((int)threadIdx.x < E) hist[(size_t)blockIdx.x * E + threadIdx.x] = run;
  if (p < P) rank[p] = rk;
}

// Step 2 of 2 (one CTA per chunk): the chunk's offset for each expert (pairs
// of that expert in all earlier chunks, plus the expert's start), then its
// pairs placed at offset + rank.  CTA 0 also writes the per-expert lists and
// marks the unused tail of the sorted list.
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_place_kernel(const int32_t* __restrict__ ids, int E, int P, const int32_t* __restrict__ emap, int G,
                       const int32_t* __restrict__ hist, const int32_t* __restrict__ rank, int n_chunks, RouteOut r,
                       int make_mtiles) {
  extern __shared__ int32_t start[];  // [E] this chunk's first position for each expert
  __shared__ int scratch[33];
  const int tid = threadIdx.x, c = blockIdx.x;
  int before = 0, tot = 0;  // expert tid's pairs in earlier chunks, in all chunks
  if (tid < E) {
    for (int cc = 0; cc < n_chunks; ++cc) {
      const int h = hist[(size_t)cc * E + tid];
      tot += h;
      before += cc < c ? h : 0;
    }
  }
  int n_valid = 0;
  int excl;
  if (c == 0) {
    excl = write_lists(tot, E, P, r, make_mtiles, scratch, &n_valid);
  } else {
    excl = block_excl_scan(tot, scratch, &n_valid);
  }
  if (tid < E) start[tid] = excl + before;
  __syncthreads();
  const int p = c * kRouteThreads + tid;
  if (p < P) {
    const int e = local_expert(ids, p, emap, G, E);
    if (e >= 0) {
      const int pos = chk(start[e] + rank[p], P, r.status);
      r.sorted_pair[pos] = p;
      r.pair_pos[p] = pos;
    } else {
      r.pair_pos[p] = -1;
    }
  }
  if (c == 0)
    for (int i = n_valid + tid; i < P; i += kRouteThreads) r.sorted_pair[i] = -1;
}

// Top-k routing from router logits, one warp per token (G <= 1024: each
// lane holds up to 32 logits in registers).  Experts are selected by logit,
// which orders them exactly as their softmax probabilities do; among equal
// logits the lower id comes first.  Weights: exp(l - max) over the sum of
// the selected ones (renormalised) or of all (softmax).
constexpr int kRouterMaxExperts = 1024;
constexpr int kRouterMaxTopk = 64;

__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T, int G, int topk,
                                                          int renorm, int32_t* __restrict__ ids,
                                                          float* __restrict__ w) {
  const int t = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + (size_t)t * G;
  float v[kRouterMaxExperts / 32];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kRouterMaxExperts / 32; ++j) {
    const int i = lane + 32 * j;
    v[j] = i < G ? row[i] : -INFINITY;
    m = fmaxf(m, v[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float all = 0.f;
#pragma unroll
  for (int j = 0; j < kRouterMaxExperts / 32; ++j)
    if (lane + 32 * j < G) all += expf(v[j] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) all += __shfl_xor_sync(0xffffffffu, all, o);
  uint32_t taken = 0;           // bit j: logit j of this lane already selected
  float ek[kRouterMaxTopk / 32] = {0.f, 0.f};  // exp(l - max) of selection k, kept by lane k % 32
  for (int k = 0; k < topk; ++k) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < kRouterMaxExperts / 32; ++j) {
      const int i = lane + 32 * j;
      if (i < G && !((taken >> j) & 1u) && (v[j] > bv || bi == 0x7FFFFFFF)) {
        bv = v[j];
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == (k & 31)) ek[k >> 5] = expf(bv - m);
    if (lane == 0) ids[(size_t)t * topk + k] = bi;
  }
  float sel = ek[0] + ek[1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, o);
  const float den = renorm ? sel : all;
  for (int k = lane; k < topk; k += 32) w[(size_t)t * topk + k] = __fdiv_rn(ek[k >> 5], den);
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int T, int G, int topk, int renorm, int32_t* ids, float* w,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (T + warps_per_block - 1) / warps_per_block;
  router_topk_kernel<<<blocks, 32 * warps_per_block, 0, s>>>(logits, T, G, topk, renorm, ids, w);
  return cudaGetLastError();
}

bool route_two_pass(long long P) { return P > kRouteThreads && P <= kRouteTwoPassMax; }

cudaError_t launch_route(const int32_t* topk_ids, int E, int T, int topk, const int32_t* emap, int G,
                         const RouteOut& r, int make_mtiles, cudaStream_t s, int32_t* hist, int32_t* rank) {
  const long long P = (long long)T * topk;
  cudaError_t err;
  if (route_two_pass(P) && hist && rank) {
    const int n_chunks = (int)((P + kRouteThreads - 1) / kRouteThreads);
    const size_t smem1 = (size_t)32 * E * sizeof(int32_t);
    err = cudaFuncSetAttribute(route_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    if (err != cudaSuccess) return err;
    route_hist_kernel<<<n_chunks, kRouteThreads, smem1, s>>>(topk_ids, E, (int)P, emap, G, hist, rank);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    route_place_kernel<<<n_chunks, kRouteThreads, (size_t)E * sizeof(int32_t), s>>>(topk_ids, E, (int)P, emap, G, hist,
                                                                                     rank, n_chunks, r, make_mtiles);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)34 * E * sizeof(int32_t);
  err = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  route_kernel<<<1, kRouteThreads, smem, s>>>(topk_ids, E, T, topk, emap, G, r, make_mtiles);
  return cudaGetLastError();
}

}  // namespace moe
