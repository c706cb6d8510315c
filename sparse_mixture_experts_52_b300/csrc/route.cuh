// Router and gating kernels.
//
// Gating follows the three forms of the pages: softmax over E -> top-k ->
// renormalise (SparseMoEGate / MoELayer), top-k on the logits -> softmax over
// the k (BEE-30064 routing steps 2-3, top_k_gating), and selection on softmax +
// per-expert bias with weights from the unbiased softmax (DeepSeek-V3).  One
// warp owns one token; lane l holds experts l, l+32, ... in registers, the
// top-k is k rounds of a warp arg-max with the lower expert index winning equal
// scores.  Load-balance partial sums (sum of softmax, top-k counts, arg-max
// counts) are kept per block in a fixed order and reduced by k_route_finalize,
// so f, P and aux are bitwise reproducible.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "groups.cuh"

namespace moe {

enum : int { ROUTE_SOFTMAX_TOPK = 0, ROUTE_TOPK_SOFTMAX = 1, ROUTE_BIASED_SOFTMAX = 2 };
enum : int { AUXF_TOPK_COUNT = 0, AUXF_ARGMAX = 1 };
constexpr int kMaxK = 16;
constexpr int kRouteWarps = 8;          // warps per routing block
constexpr int kRouteMaxBlocks = 296;    // partial-sum rows (fixed: layout must not depend on the GPU)

__host__ __device__ inline int route_blocks(int T) {
  const int nb = (T + kRouteWarps - 1) / kRouteWarps;
  return nb < 1 ? 1 : (nb > kRouteMaxBlocks ? kRouteMaxBlocks : nb);
}

struct RouteArgs {
  int T, d, E, k, route, renorm;
  const float* logit_bias;    // [E] or null
  const float* select_bias;   // [E] or null
  const float* logits_in;     // gate-from-logits: [T, ld_in]
  int ld_in;
  float* logits_out;          // [T, E] or null
  int32_t* idx;               // [T, k]
  float* w;                   // [T, k]
  float* p_part;              // [E, nb] (expert-major: one row per expert)
  int32_t* c_part;            // [E, nb] top-k counts
  int32_t* a_part;            // [E, nb] arg-max counts
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
__device__ __forceinline__ void warp_argmax(float& v, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (ov > v || (ov == v && oe < e)) {
      v = ov;
      e = oe;
    }
  }
}

// Per-lane accumulators of the load-balance statistics for experts lane+32*i.
template <int NPL>
struct LaneStats {
  float p[NPL];
  int cnt[NPL];
  int amax[NPL];
  __device__ void zero() {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      p[i] = 0.f;
      cnt[i] = 0;
      amax[i] = 0;
    }
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
        if (be == lane + 32 * i) {
          taken |= 1u << i;
          st.cnt[i] += 1;
        }
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

// Block epilogue of the statistics: warps' partials summed in warp order.
template <int NPL>
__device__ __forceinline__ void flush_stats(const LaneStats<NPL>& st, int E, float* p_part,
                                            int32_t* c_part, int32_t* a_part) {
  __shared__ float s_p[kRouteWarps][32 * NPL];
  __shared__ int s_c[kRouteWarps][32 * NPL];
  __shared__ int s_a[kRouteWarps][32 * NPL];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    s_p[warp][lane + 32 * i] = st.p[i];
    s_c[warp][lane + 32 * i] = st.cnt[i];
    s_a[warp][lane + 32 * i] = st.amax[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float ps = 0.f;
    int cs = 0, as = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      ps += s_p[w][e];
      cs += s_c[w][e];
      as += s_a[w][e];
    }
    p_part[static_cast<int64_t>(e) * gridDim.x + blockIdx.x] = ps;
    c_part[static_cast<int64_t>(e) * gridDim.x + blockIdx.x] = cs;
    a_part[static_cast<int64_t>(e) * gridDim.x + blockIdx.x] = as;
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

// Gate from precomputed logits (tensor-core router), E <= 32 * NPL.
template <int NPL>
__global__ void __launch_bounds__(kRouteWarps * 32) k_gate(const RouteArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float lb[NPL], sb[NPL];
  load_biases<NPL>(a, lane, lb, sb);
  LaneStats<NPL> st;
  st.zero();
  const int nw = gridDim.x * kRouteWarps;
  for (int t = blockIdx.x * kRouteWarps + warp; t < a.T; t += nw) {
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
  flush_stats<NPL>(st, a.E, a.p_part, a.c_part, a.a_part);
}

template <typename TE>
__device__ __forceinline__ float to_f32(TE v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Fused router + gating on the CUDA cores for E <= EP <= 64: lane l sums the
// products of d-indices l, l+32, ... for all experts (fp32 FMA), a butterfly
// all-reduce completes the E logits, then the token is gated in registers.
template <typename TE, int EP>
__global__ void __launch_bounds__(kRouteWarps * 32)
k_route_warp(const RouteArgs a, const TE* __restrict__ x, const TE* __restrict__ w_g) {
  constexpr int NPL = (EP + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float lb[NPL], sb[NPL];
  load_biases<NPL>(a, lane, lb, sb);
  LaneStats<NPL> st;
  st.zero();
  const int nw = gridDim.x * kRouteWarps;
  const int E = a.E, d = a.d;
  for (int t = blockIdx.x * kRouteWarps + warp; t < a.T; t += nw) {
    float acc[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[e] = 0.f;
    const TE* xr = x + static_cast<int64_t>(t) * d;
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
    float l[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      float v = 0.f;
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e == lane + 32 * i) v = acc[e];
      l[i] = v + lb[i];
      const int e = lane + 32 * i;
      if (a.logits_out && e < E) a.logits_out[static_cast<int64_t>(t) * E + e] = l[i];
    }
    gate_token<NPL>(l, sb, E, a.k, a.route, a.renorm, lane,
                    a.idx + static_cast<int64_t>(t) * a.k, a.w + static_cast<int64_t>(t) * a.k, st);
  }
  flush_stats<NPL>(st, E, a.p_part, a.c_part, a.a_part);
}

// f_i, P_i and aux from the per-block partials.  Block e reduces expert e's
// row (thread t sums partial rows t, t+256, ... in float64; warps then combine
// in a fixed tree), writes f[e] and P[e], and the last block to finish (a
// counter in the workspace header, reset by that block) sums f_e * P_e in
// expert order for aux.  Every sum has a fixed order: bitwise reproducible.
__global__ void __launch_bounds__(256)
k_route_finalize(int nb, int T, int E, int aux_f, float alpha, const float* p_part,
                 const int32_t* c_part, const int32_t* a_part, float* f, float* P, float* aux,
                 double* fp_scratch, unsigned int* done_counter) {
  __shared__ double s_p[8];
  __shared__ int s_c[8], s_a[8];
  __shared__ int s_last;
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(e) * nb;
  double ps = 0.0;
  int cs = 0, as = 0;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    ps += static_cast<double>(p_part[row + b]);
    cs += c_part[row + b];
    as += a_part[row + b];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ps += __shfl_xor_sync(0xffffffffu, ps, o);
    cs += __shfl_xor_sync(0xffffffffu, cs, o);
    as += __shfl_xor_sync(0xffffffffu, as, o);
  }
  if (lane == 0) {
    s_p[warp] = ps;
    s_c[warp] = cs;
    s_a[warp] = as;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ps = 0.0;
    cs = 0;
    as = 0;
    for (int w = 0; w < (blockDim.x >> 5); ++w) {
      ps += s_p[w];
      cs += s_c[w];
      as += s_a[w];
    }
    const float Pe = static_cast<float>(ps / static_cast<double>(T));
    const float fe = static_cast<float>(aux_f == AUXF_ARGMAX ? as : cs) / static_cast<float>(T);
    P[e] = Pe;
    f[e] = fe;
    fp_scratch[e] = static_cast<double>(fe) * static_cast<double>(Pe);
    __threadfence();
    s_last = (atomicAdd(done_counter, 1u) == static_cast<unsigned int>(E - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    const volatile double* fp = fp_scratch;
    double sum = 0.0;
    for (int i = 0; i < E; ++i) sum += fp[i];
    *aux = static_cast<float>(static_cast<double>(alpha) * E * sum);
    *done_counter = 0u;   // ready for the next call on this workspace
  }
}

// W_g [d, E] -> W_g^T [E_pad, d] (rows >= E zero): the K-major B operand of
// the tensor-core router.
__global__ void k_transpose_wg(const __nv_bfloat16* __restrict__ w_g, int d, int E, int E_pad,
                               __nv_bfloat16* __restrict__ wgT) {
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
