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
//                lists the taken tokens and writes the slot table [E, T]; the
//                last block reduces the statistics.
//  k_ec_gather   x_perm[r] = x[ec_token[r]] for the E*C expert-ordered rows.
//  k_ec_combine  out[t] = sum over the experts that took t (ascending) of
//                w * y[slot] + sum_s y_shared[s, t], fp32, rounded once.
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
  int32_t* offsets;          // [E + 1] = e * C
  int32_t* counts;           // [E] = C, or null
  unsigned int* done;        // last-block counter (zero between calls)
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

// Order-preserving map of a logit to an unsigned key: a larger logit gives a
// larger key, -0 and +0 give the same key and NaN gives 0 (below -inf).
__device__ __forceinline__ uint32_t ec_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (v != v) return 0u;
  if ((u & 0x7fffffffu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block e: the C-th largest key of column e by a most-significant-digit radix
// select (four 8-bit digits, a shared histogram per digit), then the taken
// tokens in ascending order: every token above that key, and the first
// `need` tokens equal to it.
__global__ void __launch_bounds__(kEcThreads) k_ec_select(const EcArgs a) {
  __shared__ unsigned int s_hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ int s_wcnt[2][kEcThreads / 32];
  griddep_wait();
  griddep_launch_dependents();
  const int e = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, C = a.C;
  const float* col = a.scoresT + static_cast<int64_t>(e) * T;

  // C == 0 takes nothing: no key exceeds 0xffffffff (NaN maps to 0) and need is 0
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
    if (warp == 0) {
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
            s_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
            s_need = need - acc;
          }
          acc += c[j];
        }
      }
    }
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
      a.ec_token[row] = t;
      a.ec_w[row] = expf(v - a.tok_max[t]) / a.tok_sum[t];   // the token's softmax p[t, e]
    }
    if (valid) a.ec_slot[static_cast<int64_t>(e) * T + t] = take ? static_cast<int32_t>(row) : -1;
    eq_carry += eq_total;
    take_carry += take_total;
    __syncthreads();   // s_wcnt is rewritten by the next chunk
  }
  if (tid == 0) {
    a.offsets[e + 1] = (e + 1) * C;
    if (e == 0) a.offsets[0] = 0;
    if (a.counts) a.counts[e] = C;
  }
  if (arrive_last_block(a.done)) {
    __shared__ int s_cnt[kMaxExperts];
    for (int i = tid; i < a.E; i += blockDim.x) s_cnt[i] = C;
    __syncthreads();
    stats_finalize(a.st, s_cnt);
    if (tid == 0) *a.done = 0u;   // ready for the next grid on this workspace
  }
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

// out[t] = sum over e ascending with ec_slot[e, t] >= 0 of ec_w[slot] * y[slot]
//          + sum_s y_shared[s, t]; warp per token, fp32 sums, one rounding.
// Lane l holds the slots of experts l, l + 32, ... (E <= 32 * kEcMaxNJ).
constexpr int kEcMaxNJ = kMaxExperts / 32;

template <typename TE>
__global__ void __launch_bounds__(256)
k_ec_combine(const TE* __restrict__ y, const int32_t* __restrict__ ec_slot,
             const float* __restrict__ ec_w, const TE* __restrict__ y_shared, int n_shared,
             int T, int E, int d, TE* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nchunk = d / 8;
  const int nj = (E + 31) / 32;
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += nw) {
    int slot[kEcMaxNJ];
    float wt[kEcMaxNJ];
#pragma unroll
    for (int j = 0; j < kEcMaxNJ; ++j) {
      const int e = lane + 32 * j;
      slot[j] = (j < nj && e < E) ? __ldg(ec_slot + static_cast<int64_t>(e) * T + t) : -1;
      wt[j] = slot[j] >= 0 ? __ldg(ec_w + slot[j]) : 0.f;
    }
    constexpr int U = 2;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
#pragma unroll
      for (int j = 0; j < kEcMaxNJ; ++j) {
        if (j >= nj) break;
        unsigned int taken = __ballot_sync(0xffffffffu, slot[j] >= 0);
        while (taken) {
          const int b = __ffs(taken) - 1;
          taken &= taken - 1u;
          const int s = __shfl_sync(0xffffffffu, slot[j], b);
          const float w = __shfl_sync(0xffffffffu, wt[j], b);
          float v[U][8];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int c = c0 + lane + 32 * u;
            if (c < nchunk) load8(y + static_cast<int64_t>(s) * d + c * 8, v[u]);
          }
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = fmaf(w, v[u][i], acc[u][i]);
        }
      }
      for (int s = 0; s < n_shared; ++s) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + lane + 32 * u;
          if (c < nchunk) {
            float v[8];
            load8(y_shared + (static_cast<int64_t>(s) * T + t) * d + c * 8, v);
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
