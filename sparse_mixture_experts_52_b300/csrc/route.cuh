// Router, gating, load-balance statistics and the dispatch bookkeeping.
//
// Gating follows the three forms of the pages: softmax over E -> top-k ->
// renormalise (SparseMoEGate / MoELayer), top-k on the logits -> softmax over
// the k (BEE-30064 routing steps 2-3, top_k_gating), and selection on softmax +
// per-expert bias with weights from the unbiased softmax (DeepSeek-V3).  One
// warp owns one token; lane l holds experts l, l+32, ... in registers, the
// top-k is k rounds of a warp arg-max with the lower expert index winning equal
// scores.
//
// A routing grid gives each block a contiguous range of 32-token chunks.
// After gating its tokens, the block ranks every assignment (t, j) inside its
// chunk among the chunk's assignments to the same expert, in ascending t*k+j
// (a token's k experts are distinct, so this is the number of earlier tokens
// of the chunk routed to that expert), stores the chunk's count per expert,
// and adds those counts to per-expert totals with integer atomics (whose sum
// does not depend on their order).  The last block to finish (a
// self-resetting counter in the workspace) turns the totals into counts, kept
// = min(count, C) and offsets, and sums the per-block softmax partials into
// P, f and aux in a fixed order.  The permute kernel later adds, for each
// token, the counts of the earlier chunks to the in-chunk rank: the stable
// rank of the assignment inside its expert.  Every result is bitwise
// reproducible.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "groups.cuh"
#include "ptx_sm100.cuh"

namespace moe {

enum : int { ROUTE_SOFTMAX_TOPK = 0, ROUTE_TOPK_SOFTMAX = 1, ROUTE_BIASED_SOFTMAX = 2 };
enum : int { AUXF_TOPK_COUNT = 0, AUXF_ARGMAX = 1 };
enum : int { DEV_ERR_BAD_EXPERT_INDEX = 8 };   // status bit: an expert index outside [0, E)
constexpr int kMaxK = 16;
constexpr int kRouteWarps = 8;          // warps per routing block
constexpr int kRouteThreads = kRouteWarps * 32;
constexpr int kGateWarps = 16;          // warps per block of the gate-from-logits grid
constexpr int kRouteMaxBlocks = 296;    // partial-sum rows (fixed: layout must not depend on the GPU)
constexpr int kSmallRouteMaxT = 512;   // the block-per-token router takes T <= this
constexpr int kChunk = 32;              // tokens per ranking chunk (one warp's lanes)
constexpr int kRouteMaxRows = 512;      // routing-grid blocks whose softmax partials the header holds

__host__ __device__ inline int num_chunks(int T) { return (T + kChunk - 1) / kChunk; }
// row stride of the per-chunk counts: a multiple of 32 chunks (128 bytes)
__host__ __device__ inline int chunk_stride(int T) { return (num_chunks(T) + 31) / 32 * 32; }
// chunks per routing block, and the number of blocks
__host__ __device__ inline int route_cpb(int T) {
  const int nc = num_chunks(T) < 1 ? 1 : num_chunks(T);
  return (nc + kRouteMaxBlocks - 1) / kRouteMaxBlocks;
}
__host__ __device__ inline int route_blocks(int T) {
  const int nc = num_chunks(T) < 1 ? 1 : num_chunks(T);
  const int cpb = route_cpb(T);
  return (nc + cpb - 1) / cpb;
}

struct DispatchArgs {
  int T, k, E, C;          // C = INT_MAX when there is no capacity limit
  int cpb;                 // chunks per block
  int32_t* crank;          // [T*k] in-chunk rank of each assignment
  int32_t* hist;           // [E, chunk_stride(T)] per-chunk counts
  int32_t* totals;         // [E] assignments per expert (zero between calls)
  int32_t* counts;         // [E]
  int32_t* kept;           // [E]
  int32_t* offsets;        // [E+1]
  unsigned int* done;      // self-resetting block counter (starts at 0)
  int* err;                // device status word
};

struct RouteArgs {
  int T, d, E, k, route, renorm;
  const float* logit_bias;    // [E] or null
  const float* select_bias;   // [E] or null
  const float* logits_in;     // gate-from-logits: [T, ld_in]
  int ld_in;
  float* logits_out;          // [T, E] or null
  int32_t* idx;               // [T, k]
  float* w;                   // [T, k]
  float* p_part;              // [E + 1, nb] per-block sums of the softmax (expert-major), row E:
                              // sums of logsumexp^2 (router z-loss); zero between calls
  unsigned int* a_tot;        // [E] arg-max counts (zero between calls)
  int aux_f;
  float alpha;
  float* f;                   // [E]
  float* P;                   // [E]
  float* aux;                 // [1]
  float* z;                   // [1] router z-loss, or null
  DispatchArgs dp;
};

// The statistics reduction: P, f and aux from the routing grid's per-block
// softmax partials (p_part, nb blocks), arg-max totals and counts.
struct StatsArgs {
  float* p_part;              // [E + 1, nb]; cleared after reading
  int nb;
  unsigned int* a_tot;        // [E]; cleared after reading
  const int32_t* counts;      // [E] assignments per expert (when count_all < 0)
  int count_all;              // >= 0: every expert has this many (Expert Choice)
  int T, E, aux_f;
  float alpha;
  float* f;
  float* P;
  float* aux;
  float* z;                   // router z-loss, or null
  unsigned int* done;         // last-block counter of the reduction (zero between calls)
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// arg-max over the warp: larger value wins, the smaller index wins equal values
// Order-preserving map of a (non-NaN) float to an unsigned key: a larger
// value gives a larger key, -0 and +0 the same one.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp-wide (largest v, lowest e among equal v): two warp reductions
// (redux.sync) instead of a five-step shuffle tree of value-index pairs.
// v must not be NaN (the callers rank NaN as -inf).
__device__ __forceinline__ void warp_argmax(float& v, int& e) {
  const uint32_t key = order_key(v);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  const uint32_t cand = (key == kmax) ? static_cast<uint32_t>(e) : 0xffffffffu;
  e = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
  v = __uint_as_float((kmax & 0x80000000u) ? (kmax & 0x7fffffffu) : ~kmax);
}

// Per-lane accumulators of the load-balance statistics for experts lane+32*i.
template <int NPL>
struct LaneStats {
  float p[NPL];
  int amax[NPL];
  float z;   // lane 0: sum over the warp's tokens of logsumexp(logits)^2
  __device__ void zero() {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      p[i] = 0.f;
      amax[i] = 0;
    }
    z = 0.f;
  }
};

// Gates one token.  l[i] is the logit of expert lane + 32*i (anything for
// experts >= E), already including logit_bias.  sb[i] is that expert's
// selection bias.  Writes idx/w of the token (lanes j < k write slot j).
template <int NPL>
__device__ __forceinline__ void gate_token(const float (&l)[NPL], const float (&sb)[NPL],
                                           int E, int k, int route, int renorm, int lane,
                                           int32_t* idx_out, float* w_out, LaneStats<NPL>& st) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  float lv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    const float v = l[i];
    lv[i] = (e < E && v == v) ? v : NEG_INF;   // NaN logits rank last
  }
  float m = NEG_INF;
#pragma unroll
  for (int i = 0; i < NPL; ++i) m = fmaxf(m, lv[i]);
  m = warp_max(m);
  float p[NPL];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    p[i] = (e < E) ? expf(lv[i] - m) : 0.f;
    s += p[i];
  }
  s = warp_sum(s);
#pragma unroll
  for (int i = 0; i < NPL; ++i) p[i] = p[i] / s;
  if (lane == 0) {   // router z-loss term: logsumexp of the logits, squared
    const float lse = m + logf(s);
    st.z += lse * lse;
  }

  // arg-max of the logits (Switch f_i)
  {
    float bv = NEG_INF;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && (be == 0x7fffffff || lv[i] > bv)) {
        bv = lv[i];
        be = e;
      }
    }
    warp_argmax(bv, be);
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (be == lane + 32 * i) st.amax[i] += 1;
  }

  float sc[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    float v = (route == ROUTE_TOPK_SOFTMAX) ? lv[i]
              : (route == ROUTE_BIASED_SOFTMAX) ? p[i] + sb[i]
                                                : p[i];
    sc[i] = (e < E && v == v) ? v : NEG_INF;
  }

  uint32_t taken = 0;
  int sel_e[kMaxK];
  float sel_v[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    sel_e[j] = 0;
    sel_v[j] = 0.f;
    if (j < k) {
      float bv = NEG_INF;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (be == 0x7fffffff || sc[i] > bv)) {
          bv = sc[i];
          be = e;
        }
      }
      warp_argmax(bv, be);
      float mine = 0.f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        if (be == lane + 32 * i) taken |= 1u << i;
        if (i == (be >> 5)) mine = (route == ROUTE_TOPK_SOFTMAX) ? lv[i] : p[i];
      }
      sel_e[j] = be;
      sel_v[j] = __shfl_sync(0xffffffffu, mine, be & 31);
    }
  }

  float w[kMaxK];
  if (route == ROUTE_TOPK_SOFTMAX) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      w[j] = (j < k) ? expf(sel_v[j] - sel_v[0]) : 0.f;
      sum += w[j];
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) w[j] = w[j] / sum;
  } else if (route == ROUTE_BIASED_SOFTMAX || renorm) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) sum += (j < k) ? sel_v[j] : 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) w[j] = sel_v[j] / sum;
  } else {
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) w[j] = sel_v[j];
  }
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k && lane == j) {
      idx_out[j] = sel_e[j];
      w_out[j] = w[j];
    }
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) st.p[i] += p[i];
}

// Block epilogue of the statistics: warps' softmax partials summed in warp
// order into column blockIdx.x of the expert-major [E, gridDim.x] partials;
// arg-max counts (integers, so their order does not matter) gathered with
// shared atomics and added to the per-expert totals.
template <int NPL, int WARPS = kRouteWarps>
__device__ __forceinline__ void flush_stats(const LaneStats<NPL>& st, int E, float* p_part,
                                            unsigned int* a_tot) {
  __shared__ float s_p[WARPS][32 * NPL];
  __shared__ int s_a[32 * NPL];
  __shared__ float s_z[WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * NPL; i += blockDim.x) s_a[i] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    s_p[warp][lane + 32 * i] = st.p[i];
    if (st.amax[i]) atomicAdd(&s_a[lane + 32 * i], st.amax[i]);
  }
  if (lane == 0) s_z[warp] = st.z;
  __syncthreads();
  if (threadIdx.x == 0) {   // z-loss row of the partials, warps in order
    float zs = 0.f;
    for (int w = 0; w < WARPS; ++w) zs += s_z[w];
    if (zs != 0.f) atomicAdd(p_part + static_cast<int64_t>(E) * gridDim.x + blockIdx.x, zs);
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float ps = 0.f;
    for (int w = 0; w < WARPS; ++w) ps += s_p[w][e];
    const int as = s_a[e];
    // a reduction into a slot that is zero and that only this block touches:
    // the value lands at L2 (0 + ps == ps, so the result is exact)
    if (ps != 0.f) atomicAdd(p_part + static_cast<int64_t>(e) * gridDim.x + blockIdx.x, ps);
    if (as) atomicAdd(a_tot + e, static_cast<unsigned int>(as));
  }
}

// ---------------------------------------------------------------- ranking
// Ranks the assignments of chunk `g` (tokens 32g .. 32g+31, lane = token)
// given each lane's experts e[j] (-1 for none: a token past T or an index
// outside [0, E); a token's valid experts are distinct); writes crank and the
// chunk's entries of hist, and adds its counts to the totals.  s_mask is this
// warp's zeroed [E] row of token masks: bit l of s_mask[x] says that the
// chunk's token l chose expert x, so the rank of (t, j) among the chunk's
// assignments to e[j] is the number of lower lanes in s_mask[e[j]] and the
// chunk's count of expert x is the number of bits of s_mask[x].  s_mask is
// zero again on return.
template <int KMAX>
__device__ __forceinline__ void rank_chunk_experts(const DispatchArgs& a, const int (&e)[KMAX],
                                                   int g, int* s_mask) {
  const int lane = threadIdx.x & 31;
  const int t = g * kChunk + lane;
  const bool valid_t = t < a.T;
  unsigned int* mask = reinterpret_cast<unsigned int*>(s_mask);
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < a.k && valid_t && e[j] >= 0) atomicOr(mask + e[j], 1u << lane);
  __syncwarp();
  const unsigned int lower = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j < a.k && valid_t)
      a.crank[static_cast<int64_t>(t) * a.k + j] = e[j] >= 0 ? __popc(mask[e[j]] & lower) : 0;
  }
  __syncwarp();
  const int ncs = chunk_stride(a.T);
  for (int x = lane; x < a.E; x += 32) {
    const int c = __popc(mask[x]);
    a.hist[static_cast<int64_t>(x) * ncs + g] = c;
    if (c) atomicAdd(a.totals + x, c);
    mask[x] = 0u;
  }
  __syncwarp();
}

// The same, reading the experts of the chunk's tokens from `idx` (from L2,
// ld.cg: this grid may have just written it).  An index outside [0, E), or one
// a token's row already holds, sets the status bit and counts as no expert.
template <int KMAX>
__device__ __forceinline__ void rank_chunk(const DispatchArgs& a, const int32_t* idx, int g,
                                           int* s_hist) {
  const int lane = threadIdx.x & 31;
  const int t = g * kChunk + lane;
  int e[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    e[j] = -1;
    if (j < a.k && t < a.T) {
      const int v = __ldcg(idx + static_cast<int64_t>(t) * a.k + j);
      bool repeated = false;
#pragma unroll
      for (int jj = 0; jj < KMAX; ++jj) repeated |= (jj < j && e[jj] == v);
      if (v >= 0 && v < a.E && !repeated) {
        e[j] = v;
      } else {
        atomicOr(a.err, DEV_ERR_BAD_EXPERT_INDEX);
      }
    }
  }
  rank_chunk_experts<KMAX>(a, e, g, s_hist);
}

// Ranks chunks [g0, g1) (warp w takes chunks g0+w, g0+w+WARPS, ...).
template <int KMAX, int WARPS = kRouteWarps>
__device__ __forceinline__ void rank_chunks(const DispatchArgs& a, const int32_t* idx, int g0,
                                            int g1) {
  __shared__ int s_hist[WARPS][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int x = lane; x < a.E; x += 32) s_hist[warp][x] = 0;
  __syncwarp();
  for (int g = g0 + warp; g < g1; g += WARPS) rank_chunk<KMAX>(a, idx, g, s_hist[warp]);
}

// Ranks every chunk of this block's range.
template <int KMAX, int WARPS = kRouteWarps>
__device__ __forceinline__ void rank_block_chunks(const DispatchArgs& a, const int32_t* idx) {
  const int g0 = blockIdx.x * a.cpb;
  rank_chunks<KMAX, WARPS>(a, idx, g0, min(g0 + a.cpb, num_chunks(a.T)));
}

// True in the one block that arrives last; every thread of the block must call
// it.  The barrier orders all of this block's writes before thread 0's
// acquire-release increment of the counter (release is cumulative over what
// the barrier made visible to thread 0); the last block's increment acquires
// every other block's writes, and its closing barrier passes them on to the
// block's threads.
__device__ __forceinline__ bool arrive_last_block(unsigned int* done) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(done)
                 : "memory");
    s_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  return s_last != 0;
}

// Last block of a routing or ranking grid: counts (from the totals, which it
// clears for the next call), kept and offsets.  Leaves the counts in s_cnt
// (shared, >= E entries).
__device__ void dispatch_finalize(const DispatchArgs& a, int* s_cnt) {
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    s_cnt[e] = __ldcg(a.totals + e);
    a.totals[e] = 0;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int run = 0;
    for (int base = 0; base < a.E; base += 32) {
      const int x = base + lane;
      const int c = x < a.E ? s_cnt[x] : 0;
      const int kp = c < a.C ? c : a.C;
      int w = kp;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      if (x < a.E) {
        a.counts[x] = c;
        a.kept[x] = kp;
        a.offsets[x] = run + w - kp;
      }
      run += __shfl_sync(0xffffffffu, w, 31);
    }
    if (lane == 0) a.offsets[a.E] = run;
  }
  __syncthreads();
}

// The statistics reduction: P, f, aux and the z-loss from the routing grid's
// per-block partials, fp32 throughout (the FP64 pipe of this GPU is 64x
// slower) and in a fixed order.  It runs on a few blocks in parallel (extra
// blocks of the permute or select grid, or its own small grid): each warp
// takes whole rows of the partials - expert rows, then the z-loss row - and
// lane l sums blocks l, l+32, ... in ascending order with every load of the
// row in flight together, a fixed shuffle tree combining the lanes.  The last
// block to finish adds aux = alpha * E * sum_e f_e P_e.
constexpr int kStatsMaxSteps = (kRouteMaxBlocks > kSmallRouteMaxT ? kRouteMaxBlocks
                                                                   : kSmallRouteMaxT) / 32 + 1;

// Blocks of `warps` warps that the reduction of E experts takes.
__host__ __device__ inline int stats_blocks(int E, int warps) {
  return (E + 1 + warps - 1) / warps;
}

__device__ __forceinline__ void stats_row(const StatsArgs& a, int r, int lane) {
  const int nb = a.nb, steps = (nb + 31) / 32;
  float* row = a.p_part + static_cast<int64_t>(r) * nb;
  float pv[kStatsMaxSteps];
#pragma unroll
  for (int s = 0; s < kStatsMaxSteps; ++s) {
    const int b = s * 32 + lane;
    pv[s] = (s < steps && b < nb) ? __ldcg(row + b) : 0.f;
  }
  // the zeroing stores after every load of the row: a store between two loads
  // would order the second load behind it
#pragma unroll
  for (int s = 0; s < kStatsMaxSteps; ++s) {
    const int b = s * 32 + lane;
    if (s < steps && b < nb) row[b] = 0.f;   // zero for the next call
  }
  float p = 0.f;
#pragma unroll
  for (int s = 0; s < kStatsMaxSteps; ++s) p += pv[s];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
  if (lane != 0) return;
  if (r == a.E) {   // the z-loss row
    if (a.z) *a.z = p / static_cast<float>(a.T);
    return;
  }
  int cnt;
  if (a.aux_f == AUXF_ARGMAX) {
    cnt = static_cast<int>(__ldcg(a.a_tot + r));
    a.a_tot[r] = 0u;   // cleared for the next call
  } else {
    cnt = a.count_all >= 0 ? a.count_all : __ldcg(a.counts + r);
  }
  a.P[r] = p / static_cast<float>(a.T);
  a.f[r] = static_cast<float>(cnt) / static_cast<float>(a.T);
}

// Block sb of the nblk blocks of the reduction.
__device__ void stats_reduce(const StatsArgs& a, int sb, int nblk) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int r = sb * nwarps + warp; r <= a.E; r += nblk * nwarps) stats_row(a, r, lane);
  if (a.aux_f != AUXF_ARGMAX) {   // arg-max totals unused: clear them for the next call
    for (int e = sb * blockDim.x + threadIdx.x; e < a.E; e += nblk * blockDim.x) a.a_tot[e] = 0u;
  }
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(a.done)
                 : "memory");
    s_last = (prev == static_cast<unsigned int>(nblk) - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  if (warp == 0) {   // aux: lane-strided over the experts, then a fixed tree
    float sum = 0.f;
    for (int e = lane; e < a.E; e += 32) sum += __ldcg(a.f + e) * __ldcg(a.P + e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      *a.aux = a.alpha * static_cast<float>(a.E) * sum;
      *a.done = 0u;   // ready for the next call on this workspace
    }
  }
}

// The reduction as a grid of its own (stats_blocks(E, 8) blocks of 256).
__global__ void __launch_bounds__(256) k_stats(const StatsArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  stats_reduce(a, blockIdx.x, gridDim.x);
}

// Common tail of the routing kernels: statistics partials, chunk ranking, and
// the last block's dispatch finalize (the statistics are reduced by a later
// grid: stats_reduce).
template <int NPL, int KMAX, int WARPS = kRouteWarps>
__device__ __forceinline__ void route_block_tail(const RouteArgs& a, const LaneStats<NPL>& st) {
  flush_stats<NPL, WARPS>(st, a.E, a.p_part, a.a_tot);
  __syncthreads();   // this block's idx writes are visible to all its warps
  rank_block_chunks<KMAX, WARPS>(a.dp, a.idx);
  if (arrive_last_block(a.dp.done)) {
    __shared__ int s_cnt[kMaxExperts];
    dispatch_finalize(a.dp, s_cnt);
    if (threadIdx.x == 0) *a.dp.done = 0u;   // ready for the next grid on this workspace
  }
}

template <int NPL>
__device__ __forceinline__ void load_biases(const RouteArgs& a, int lane, float (&lb)[NPL],
                                            float (&sb)[NPL]) {
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    lb[i] = (a.logit_bias && e < a.E) ? a.logit_bias[e] : 0.f;
    sb[i] = (a.select_bias && e < a.E) ? a.select_bias[e] : 0.f;
  }
}

template <typename TE>
__device__ __forceinline__ float to_f32(TE v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Gate from precomputed logits (tensor-core router), E <= 32 * NPL.  WARPS
// warps a block: a warp gates one token at a time, and the gating of a wide
// router (E = 256, k = 8) is a chain of shuffles, so more warps per SM hide
// its latency.
template <int NPL, int KMAX, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) k_gate(const RouteArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float lb[NPL], sb[NPL];
  load_biases<NPL>(a, lane, lb, sb);
  LaneStats<NPL> st;
  st.zero();
  const int t0 = blockIdx.x * a.dp.cpb * kChunk;
  const int t1 = min(t0 + a.dp.cpb * kChunk, a.T);
  for (int t = t0 + warp; t < t1; t += WARPS) {
    float l[NPL];
    const float* row = a.logits_in + static_cast<int64_t>(t) * a.ld_in;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      l[i] = (e < a.E) ? row[e] + lb[i] : 0.f;
      if (a.logits_out && e < a.E) a.logits_out[static_cast<int64_t>(t) * a.E + e] = l[i];
    }
    gate_token<NPL>(l, sb, a.E, a.k, a.route, a.renorm, lane,
                    a.idx + static_cast<int64_t>(t) * a.k, a.w + static_cast<int64_t>(t) * a.k, st);
  }
  route_block_tail<NPL, KMAX, WARPS>(a, st);
}

// Router logits of one token on the CUDA cores for E <= EP <= 64: lane l sums
// the products of d-indices l, l+32, ... for all experts (fp32 FMA), a
// butterfly all-reduce completes the E sums; l[i] is the logit of expert
// lane + 32*i plus lb[i].
template <typename TE, int EP>
__device__ __forceinline__ void warp_logits(const TE* __restrict__ xr, const TE* __restrict__ w_g,
                                            int d, int E, int lane,
                                            const float (&lb)[(EP + 31) / 32],
                                            float (&l)[(EP + 31) / 32]) {
  constexpr int NPL = (EP + 31) / 32;
  float acc[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int i = lane; i < d; i += 32) {
    const float xv = to_f32<TE>(xr[i]);
    const TE* wr = w_g + static_cast<int64_t>(i) * E;
#pragma unroll
    for (int e = 0; e < EP; ++e)
      if (e < E) acc[e] = fmaf(xv, to_f32<TE>(wr[e]), acc[e]);
  }
#pragma unroll
  for (int e = 0; e < EP; ++e) acc[e] = warp_sum(acc[e]);
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    float v = 0.f;
#pragma unroll
    for (int e = 0; e < EP; ++e)
      if (e == lane + 32 * i) v = acc[e];
    l[i] = v + lb[i];
  }
}

// Fused router + gating on the CUDA cores for E <= EP <= 64: the logits of
// each token (warp_logits), then the token is gated in registers.
template <typename TE, int EP, int KMAX>
__global__ void __launch_bounds__(kRouteThreads)
k_route_warp(const RouteArgs a, const TE* __restrict__ x, const TE* __restrict__ w_g) {
  constexpr int NPL = (EP + 31) / 32;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float lb[NPL], sb[NPL];
  load_biases<NPL>(a, lane, lb, sb);
  LaneStats<NPL> st;
  st.zero();
  const int E = a.E, d = a.d;
  const int t0 = blockIdx.x * a.dp.cpb * kChunk;
  const int t1 = min(t0 + a.dp.cpb * kChunk, a.T);
  for (int t = t0 + warp; t < t1; t += kRouteWarps) {
    float l[NPL];
    warp_logits<TE, EP>(x + static_cast<int64_t>(t) * d, w_g, d, E, lane, lb, l);
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (a.logits_out && e < E) a.logits_out[static_cast<int64_t>(t) * E + e] = l[i];
    }
    gate_token<NPL>(l, sb, E, a.k, a.route, a.renorm, lane,
                    a.idx + static_cast<int64_t>(t) * a.k, a.w + static_cast<int64_t>(t) * a.k, st);
  }
  route_block_tail<NPL, KMAX>(a, st);
}

// Router + gating for short batches (T <= kSmallRouteMaxT), E <= EP <= 64:
// one block per token.  When E is a multiple of VE (the experts in 16 bytes),
// thread (g, s) of the block takes expert group g (VE consecutive experts,
// one 16-byte load per row of W_g) and the d-indices s, s+S, ...; otherwise
// thread i takes the 16-byte vectors i, i+256, ... of x with scalar loads of
// the matching W_g rows.  fp32 FMA, a block reduction in a fixed order
// completes the E logits, warp 0 gates the token.  The last block ranks every
// chunk of the batch and finalises.

template <typename TE, int EP, int KMAX>
__global__ void __launch_bounds__(kRouteThreads)
k_route_small(const RouteArgs a, const TE* __restrict__ x, const TE* __restrict__ w_g) {
  constexpr int NPL = (EP + 31) / 32;
  constexpr int VE = 16 / static_cast<int>(sizeof(TE));   // elements per 16 bytes
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float s_red[kRouteWarps][EP];
  __shared__ float s_logit[EP];
  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, d = a.d;
  const TE* xr = x + static_cast<int64_t>(t) * d;
  if (E % VE == 0) {
    const int G = E / VE;
    int Gp = 1;
    while (Gp < G) Gp <<= 1;
    const int S = kRouteThreads / Gp;        // threads per expert group
    const int g = tid / S, sl = tid % S;
    float acc[VE];
#pragma unroll
    for (int v = 0; v < VE; ++v) acc[v] = 0.f;
    if (g < G) {
#pragma unroll 4
      for (int i = sl; i < d; i += S) {
        const float xv = to_f32<TE>(__ldg(xr + i));
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(w_g + static_cast<int64_t>(i) * E + g * VE));
        const TE* wp = reinterpret_cast<const TE*>(&wv);
#pragma unroll
        for (int v = 0; v < VE; ++v) acc[v] = fmaf(xv, to_f32<TE>(wp[v]), acc[v]);
      }
    }
    const int W = S < 32 ? S : 32;           // lanes of one group inside a warp
    for (int o = W >> 1; o > 0; o >>= 1) {
#pragma unroll
      for (int v = 0; v < VE; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], o);
    }
    if (lane % W == 0) {
#pragma unroll
      for (int v = 0; v < VE; ++v) s_red[warp][(lane / W) * VE + v] = acc[v];
    }
    __syncthreads();
    if (tid < E) {
      const int ge = tid / VE, v = tid % VE;
      float sum = 0.f;
      if (S >= 32) {
        for (int w = ge * S / 32; w < (ge + 1) * S / 32; ++w) sum += s_red[w][v];
      } else {
        sum = s_red[(ge * S) / 32][(((ge * S) % 32) / S) * VE + v];
      }
      s_logit[tid] = sum;
    }
  } else {
    float acc[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[e] = 0.f;
    for (int i0 = tid * VE; i0 < d; i0 += blockDim.x * VE) {
      const uint4 xv4 = __ldg(reinterpret_cast<const uint4*>(xr + i0));
      const TE* xs = reinterpret_cast<const TE*>(&xv4);
#pragma unroll
      for (int u = 0; u < VE; ++u) {
        const float xv = to_f32<TE>(xs[u]);
        const TE* wr = w_g + static_cast<int64_t>(i0 + u) * E;
#pragma unroll
        for (int e = 0; e < EP; ++e)
          if (e < E) acc[e] = fmaf(xv, to_f32<TE>(__ldg(wr + e)), acc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      const float v = warp_sum(acc[e]);
      if (lane == 0) s_red[warp][e] = v;
    }
    __syncthreads();
    if (tid < E) {
      float sum = 0.f;
      for (int w = 0; w < kRouteWarps; ++w) sum += s_red[w][tid];
      s_logit[tid] = sum;
    }
  }
  __syncthreads();
  LaneStats<NPL> st;
  st.zero();
  if (warp == 0) {
    float lb[NPL], sb[NPL];
    load_biases<NPL>(a, lane, lb, sb);
    float l[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      l[i] = (e < E ? s_logit[e] : 0.f) + lb[i];
      if (a.logits_out && e < E) a.logits_out[static_cast<int64_t>(t) * E + e] = l[i];
    }
    gate_token<NPL>(l, sb, E, a.k, a.route, a.renorm, lane,
                    a.idx + static_cast<int64_t>(t) * a.k, a.w + static_cast<int64_t>(t) * a.k, st);
  }
  flush_stats<NPL>(st, E, a.p_part, a.a_tot);
  if (arrive_last_block(a.dp.done)) {
    __shared__ int s_cnt[kMaxExperts];
    rank_chunks<KMAX>(a.dp, a.idx, 0, num_chunks(a.T));
    __syncthreads();
    dispatch_finalize(a.dp, s_cnt);
    if (threadIdx.x == 0) *a.dp.done = 0u;
  }
}

// Ranking of caller-supplied expert indices (the standalone dispatch entry
// points): the same chunk ranks, prefixes, counts, kept and offsets as the
// routing kernels produce.
template <int KMAX>
__global__ void __launch_bounds__(kRouteThreads) k_dispatch_rank(const DispatchArgs a,
                                                                 const int32_t* idx) {
  griddep_wait();
  griddep_launch_dependents();
  rank_block_chunks<KMAX>(a, idx);
  if (arrive_last_block(a.done)) {
    __shared__ int s_cnt[kMaxExperts];
    dispatch_finalize(a, s_cnt);
    if (threadIdx.x == 0) *a.done = 0u;
  }
}

// W_g [d, E] -> W_g^T [E_pad, d] (rows >= E zero): the K-major B operand of
// the tensor-core router.
__global__ void k_transpose_wg(const __nv_bfloat16* __restrict__ w_g, int d, int E, int E_pad,
                               __nv_bfloat16* __restrict__ wgT) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ __nv_bfloat16 tile[32][33];
  const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int i = i0 + r, e = e0 + threadIdx.x;
    tile[r][threadIdx.x] = (i < d && e < E) ? w_g[static_cast<int64_t>(i) * E + e]
                                            : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int e = e0 + r, i = i0 + threadIdx.x;
    if (e < E_pad && i < d) wgT[static_cast<int64_t>(e) * d + i] = tile[threadIdx.x][r];
  }
}

}  // namespace moe
