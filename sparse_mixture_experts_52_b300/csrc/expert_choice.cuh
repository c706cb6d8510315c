// Expert Choice routing: every expert takes the C tokens with the largest
// router logits of its column (lower token first among equal logits), so each
// expert processes exactly C rows; a token may be taken by several experts or
// by none.  The gate weight of a taken (token, expert) pair is the token's
// softmax probability over the experts.  ("AI-Research-SKILLs MoE 训练实战…全指南"
// §4.2 Expert Choice; "第7章 Mixture of Experts" §7.2.)
//
//  k_ec_scores   warp per token: logits (on the CUDA cores, or read from the
//                tensor-core router), written expert-major [E, T]; the token's
//                softmax maximum and sum; softmax and z-loss partials for the
//                statistics.
//  k_ec_select   block per expert: radix select of the C-th largest logit of
//                the column, then one pass in ascending token order that
//                lists the taken tokens and writes the slot table [E, T]; one
//                extra block reduces the statistics meanwhile
//                (k_ec_select_reg keeps a column of up to 8192 tokens in
//                registers).
//  k_ec_gather   x_perm[r] = x[ec_token[r]] for the E*C expert-ordered rows.
//  k_ec_combine  out[t] = sum over the experts that took t (ascending) of
//                w * y[slot] + sum_s y_shared[s, t], fp32, rounded once; in a
//                whole-layer pass the weights come from an [E, T] copy that
//                k_ec_select writes beside the slot table.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "dispatch.cuh"
#include "route.cuh"

namespace moe {

constexpr int kEcThreads = 512;

struct EcArgs {
  int T, d, E, C;
  const float* logit_bias;   // [E] or null
  const float* logits_in;    // [T, ld_in] tensor-core router output, or null
  int ld_in;
  float* logits_out;         // [T, E] or null
  float* scoresT;            // [E, T] logits, expert-major
  float* tok_max;            // [T] largest logit of each token
  float* tok_sum;            // [T] sum over experts of exp(logit - tok_max)
  int32_t* ec_token;         // [E, C] taken tokens of each expert, ascending
  float* ec_w;               // [E, C] their gate weights
  int32_t* ec_slot;          // [E, T] row e*C + r of (t, e), or -1
  float* ec_wt;              // [E, T] gate weight of (t, e) where taken (else unspecified)
  int32_t* offsets;          // [E + 1] = e * C
  int32_t* counts;           // [E] = C, or null
  StatsArgs st;              // p_part, a_tot, nb = grid of k_ec_scores, outputs
};

// Softmax, log-sum-exp, z-loss term and arg-max of one token whose logits
// (bias included) lane + 32*i holds in l[i]; the logits go out expert-major.
template <int NPL>
__device__ __forceinline__ void ec_token(const EcArgs& a, int t, int lane, const float (&l)[NPL],
                                         LaneStats<NPL>& st) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int E = a.E;
  float lv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    lv[i] = (e < E && l[i] == l[i]) ? l[i] : NEG_INF;   // NaN logits rank last
    if (e < E) {
      a.scoresT[static_cast<int64_t>(e) * a.T + t] = l[i];
      if (a.logits_out) a.logits_out[static_cast<int64_t>(t) * E + e] = l[i];
    }
  }
  float m = NEG_INF;
#pragma unroll
  for (int i = 0; i < NPL; ++i) m = fmaxf(m, lv[i]);
  m = warp_max(m);
  float p[NPL];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    p[i] = (lane + 32 * i < E) ? expf(lv[i] - m) : 0.f;
    s += p[i];
  }
  s = warp_sum(s);
#pragma unroll
  for (int i = 0; i < NPL; ++i) st.p[i] += p[i] / s;
  if (lane == 0) {
    a.tok_max[t] = m;
    a.tok_sum[t] = s;
    const float lse = m + logf(s);
    st.z += lse * lse;
  }
  // arg-max of the logits (f_i of the arg-max form), lowest expert on ties
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

// Logits on the CUDA cores (E <= EP <= 64), or from the tensor-core router's
// [T, ld_in] output when EP == 0 (then E <= 32 * NPL).
template <typename TE, int EP, int NPL>
__global__ void __launch_bounds__(kRouteThreads)
k_ec_scores(const EcArgs a, const TE* __restrict__ x, const TE* __restrict__ w_g) {
  static_assert(EP == 0 || NPL == (EP + 31) / 32, "lanes per expert block");
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float lb[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    lb[i] = (a.logit_bias && e < a.E) ? a.logit_bias[e] : 0.f;
  }
  LaneStats<NPL> st;
  st.zero();
  for (int t = blockIdx.x * kRouteWarps + warp; t < a.T; t += gridDim.x * kRouteWarps) {
    float l[NPL];
    if constexpr (EP == 0) {
      const float* row = a.logits_in + static_cast<int64_t>(t) * a.ld_in;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        l[i] = (e < a.E) ? row[e] + lb[i] : 0.f;
      }
    } else {
      warp_logits<TE, EP>(x + static_cast<int64_t>(t) * a.d, w_g, a.d, a.E, lane, lb, l);
    }
    ec_token<NPL>(a, t, lane, l, st);
  }
  flush_stats<NPL>(st, a.E, a.st.p_part, a.st.a_tot);
}

// Key of a logit for the selection: order_key, and 0 (below -inf) for NaN.
__device__ __forceinline__ uint32_t ec_key(float v) { return v != v ? 0u : order_key(v); }

// Warp 0 of a select block, after the histogram of digit `shift` of the keys
// that match `prefix`: finds the digit holding the need-th largest of them and
// publishes the longer prefix and the rank left inside it.
__device__ __forceinline__ void ec_pick_digit(const unsigned int* s_hist, int lane,
                                              uint32_t prefix, int shift, int need,
                                              uint32_t* s_prefix, int* s_need) {
  // lane l holds digits 255 - 8l .. 248 - 8l, from the top
  int c[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = static_cast<int>(s_hist[255 - 8 * lane - j]);
    sum += c[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int acc = incl - sum;   // keys in higher digits than this lane's
  if (acc < need && need <= incl) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (acc < need && need <= acc + c[j]) {
        *s_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
        *s_need = need - acc;
      }
      acc += c[j];
    }
  }
}

// Common end of both select kernels: offsets and counts of expert e.
__device__ __forceinline__ void ec_select_tail(const EcArgs& a, int e) {
  if (threadIdx.x == 0) {
    a.offsets[e + 1] = (e + 1) * a.C;
    if (e == 0) a.offsets[0] = 0;
    if (a.counts) a.counts[e] = a.C;
  }
}

// The blocks after the E select blocks reduce the routing statistics from
// the per-block partials of k_ec_scores while the others select: every expert
// has C rows (count_all), so f needs nothing from the selection.
__device__ __forceinline__ bool ec_stats_block(const EcArgs& a) {
  const int sb = static_cast<int>(blockIdx.x) - a.E;
  if (sb < 0) return false;
  stats_reduce(a.st, sb, static_cast<int>(gridDim.x) - a.E);
  return true;
}

// Block e, columns of at most kEcThreads * VPT tokens: thread i keeps the keys
// of tokens i*VPT .. i*VPT + VPT - 1 in registers.  Most-significant-digit
// radix select of the C-th largest key (four 8-bit digits; lanes that share a
// digit add to the shared histogram once, through __match_any_sync, since the
// top digit of similar logits falls into a handful of bins), then one ordered
// compaction: every token above that key and the first `need` tokens equal
// to it, positions from two block-wide exclusive scans.
template <int VPT>
__global__ void __launch_bounds__(kEcThreads) k_ec_select_reg(const EcArgs a) {
  __shared__ unsigned int s_hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ int s_wsum[kEcThreads / 32];
  griddep_wait();
  griddep_launch_dependents();
  if (ec_stats_block(a)) return;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, C = a.C;
  const float* col = a.scoresT + static_cast<int64_t>(e) * T;
  const int t0 = tid * VPT;
  uint32_t key[VPT];
  float val[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    val[v] = (t0 + v < T) ? col[t0 + v] : 0.f;
    key[v] = (t0 + v < T) ? ec_key(val[v]) : 0u;
  }
  // C == 0 takes nothing: no key exceeds 0xffffffff (NaN maps to 0) and need is 0
  uint32_t prefix = C > 0 ? 0u : 0xffffffffu, mask = 0u;
  int need = C;
  for (int shift = 24; C > 0 && shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) s_hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const bool in = (t0 + v < T) && (key[v] & mask) == prefix;
      const int bin = in ? static_cast<int>((key[v] >> shift) & 255u) : 256;
      const unsigned int peers = __match_any_sync(0xffffffffu, bin);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) ec_pick_digit(s_hist, lane, prefix, shift, need, &s_prefix, &s_need);
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
  }
  const uint32_t thr = prefix;

  // block-wide exclusive scan of one count per thread (thread order = token order)
  auto excl_scan = [&](int x) {
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int before = incl - x;
    for (int w = 0; w < warp; ++w) before += s_wsum[w];
    __syncthreads();   // s_wsum is reused by the next scan
    return before;
  };
  int n_eq = 0;
#pragma unroll
  for (int v = 0; v < VPT; ++v) n_eq += (t0 + v < T && key[v] == thr) ? 1 : 0;
  int eq_rank = excl_scan(n_eq);
  bool take[VPT];
  int n_take = 0;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const bool valid = t0 + v < T;
    const bool eq = valid && key[v] == thr;
    take[v] = (valid && key[v] > thr) || (eq && eq_rank < need);
    eq_rank += eq ? 1 : 0;
    n_take += take[v] ? 1 : 0;
  }
  int pos = excl_scan(n_take);
  const int64_t row0 = static_cast<int64_t>(e) * C;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int t = t0 + v;
    if (t >= T) break;
    if (take[v]) {
      const float w = expf(val[v] - a.tok_max[t]) / a.tok_sum[t];   // softmax p[t, e]
      a.ec_token[row0 + pos] = t;
      a.ec_w[row0 + pos] = w;
      if (a.ec_wt) a.ec_wt[static_cast<int64_t>(e) * T + t] = w;
    }
    a.ec_slot[static_cast<int64_t>(e) * T + t] = take[v] ? static_cast<int32_t>(row0 + pos) : -1;
    pos += take[v] ? 1 : 0;
  }
  ec_select_tail(a, e);
}

// The same selection for columns of any length: the column is streamed from
// memory for every digit and for the compaction, kEcThreads tokens at a time.
__global__ void __launch_bounds__(kEcThreads) k_ec_select(const EcArgs a) {
  __shared__ unsigned int s_hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ int s_wcnt[2][kEcThreads / 32];
  griddep_wait();
  griddep_launch_dependents();
  if (ec_stats_block(a)) return;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, C = a.C;
  const float* col = a.scoresT + static_cast<int64_t>(e) * T;

  uint32_t prefix = C > 0 ? 0u : 0xffffffffu, mask = 0u;
  int need = C;   // rank from the top still to find inside the keys matching prefix
  for (int shift = 24; C > 0 && shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) s_hist[i] = 0u;
    __syncthreads();
    for (int t = tid; t < T; t += blockDim.x) {
      const uint32_t k = ec_key(col[t]);
      if ((k & mask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) ec_pick_digit(s_hist, lane, prefix, shift, need, &s_prefix, &s_need);
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
  }
  const uint32_t thr = prefix;   // key of the C-th largest logit

  const unsigned int lt_mask = (1u << lane) - 1u;
  int eq_carry = 0, take_carry = 0;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + tid;
    const bool valid = t < T;
    const float v = valid ? col[t] : 0.f;
    const uint32_t k = valid ? ec_key(v) : 0u;
    const bool gt = valid && k > thr, eq = valid && k == thr;
    const unsigned int b_eq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s_wcnt[0][warp] = __popc(b_eq);
    __syncthreads();
    int eq_rank = eq_carry + __popc(b_eq & lt_mask);
    int eq_total = 0;
    for (int w = 0; w < (kEcThreads / 32); ++w) {
      if (w < warp) eq_rank += s_wcnt[0][w];
      eq_total += s_wcnt[0][w];
    }
    const bool take = gt || (eq && eq_rank < need);
    const unsigned int b_take = __ballot_sync(0xffffffffu, take);
    if (lane == 0) s_wcnt[1][warp] = __popc(b_take);
    __syncthreads();
    int pos = take_carry + __popc(b_take & lt_mask);
    int take_total = 0;
    for (int w = 0; w < (kEcThreads / 32); ++w) {
      if (w < warp) pos += s_wcnt[1][w];
      take_total += s_wcnt[1][w];
    }
    const int64_t row = static_cast<int64_t>(e) * C + pos;
    if (take) {
      const float w = expf(v - a.tok_max[t]) / a.tok_sum[t];   // the token's softmax p[t, e]
      a.ec_token[row] = t;
      a.ec_w[row] = w;
      if (a.ec_wt) a.ec_wt[static_cast<int64_t>(e) * T + t] = w;
    }
    if (valid) a.ec_slot[static_cast<int64_t>(e) * T + t] = take ? static_cast<int32_t>(row) : -1;
    eq_carry += eq_total;
    take_carry += take_total;
    __syncthreads();   // s_wcnt is rewritten by the next chunk
  }
  ec_select_tail(a, e);
}

// Row gather of the expert-ordered rows: x_perm[r] = x[ec_token[r]], warp per
// row, 16-byte vectors; block 0 also writes offsets[e] = e * C.
__global__ void __launch_bounds__(256)
k_ec_gather(const int32_t* __restrict__ ec_token, int rows, int row_bytes, int C, int E,
            const uint8_t* __restrict__ x, uint8_t* __restrict__ x_perm,
            int32_t* __restrict__ offsets) {
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = e * C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nvec = row_bytes / 16;
  for (int r = blockIdx.x * (blockDim.x >> 5) + warp; r < rows; r += nw) {
    const int t = __ldg(ec_token + r);
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(r) * row_bytes);
    for (int c = lane; c < nvec; c += 32) dst[c] = __ldg(src + c);
  }
}

// out[t] = sum over e ascending with ec_slot[e, t] >= 0 of w[e, t] * y[slot]
//          + sum_s y_shared[s, t]; fp32 sums, one rounding.  One warp per
// token: lane l reads the slots and weights of experts l, l + 32, ... (NJ
// groups of 32 experts; the two [E, T] tables side by side when the weight
// table is given, else the weights from the [E, C] list through the slots),
// then the rows of the taken experts are summed in ascending expert order,
// the loads of two experts' rows (U 16-byte vectors per lane each) in flight
// together.  TY: the expert outputs' type (the layer dtype, or fp32 for a
// bf16 layer that keeps them so); TO: the layer dtype.
template <typename TY, typename TO, int U, int NJ>
__global__ void __launch_bounds__(256, 3)
k_ec_combine(const TY* __restrict__ y, const int32_t* __restrict__ ec_slot,
             const float* __restrict__ ec_wt, const float* __restrict__ ec_w,
             const TY* __restrict__ y_shared, int n_shared, int T, int E, int d,
             TO* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nchunk = d / 8;
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += nw) {
    int slot[NJ];
    float wt[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      const int64_t at = static_cast<int64_t>(e) * T + t;
      slot[j] = e < E ? __ldg(ec_slot + at) : -1;
      if (ec_wt)
        wt[j] = e < E ? __ldg(ec_wt + at) : 0.f;
      else   // only the [E, C] weights: one more dependent load
        wt[j] = slot[j] >= 0 ? __ldg(ec_w + slot[j]) : 0.f;
    }
    for (int c0 = 0; c0 < nchunk; c0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
      constexpr int Q = 2;   // experts whose rows are loaded together
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        unsigned int taken = __ballot_sync(0xffffffffu, slot[j] >= 0);
        while (taken) {
          int s[Q];
          float w[Q];
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            s[q] = -1;
            w[q] = 0.f;
            if (taken) {
              const int b = __ffs(taken) - 1;
              taken &= taken - 1u;
              s[q] = __shfl_sync(0xffffffffu, slot[j], b);
              w[q] = __shfl_sync(0xffffffffu, wt[j], b);
            }
          }
          Raw8<TY> v[Q][U];
#pragma unroll
          for (int q = 0; q < Q; ++q)
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int c = c0 + lane + 32 * u;
              if (s[q] >= 0 && c < nchunk) v[q][u].load(y + static_cast<int64_t>(s[q]) * d + c * 8);
            }
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            if (s[q] < 0) break;
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (c0 + lane + 32 * u < nchunk) v[q][u].fma_into(w[q], acc[u]);
          }
        }
      }
      for (int sh = 0; sh < n_shared; ++sh) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + lane + 32 * u;
          if (c < nchunk) {
            float v[8];
            load8(y_shared + (static_cast<int64_t>(sh) * T + t) * d + c * 8, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] += v[i];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + lane + 32 * u;
        if (c < nchunk) store8(out + static_cast<int64_t>(t) * d + c * 8, acc[u]);
      }
    }
  }
}

}  // namespace moe
