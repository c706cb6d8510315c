// Router GEMM on the tensor cores with the gating in its epilogue, for bf16
// layers with E <= 64 experts.
//
// One CTA per 128 tokens: logits[128, E_pad] = x_tile . W_g^T accumulate in
// TMEM (tcgen05, TMA-fed ring, as in gemm_tc.cuh), then every epilogue thread
// owns one token (its TMEM lane) and gates it in registers: softmax over the
// E logits, the arg-max, the top-k by insertion in ascending expert order
// (strict comparisons, so the lower index wins equal scores), and the gate
// weights of the routing form.  The four epilogue warps hold 32 consecutive
// tokens each: exactly one ranking chunk, ranked from the registers.  The
// softmax column sums of the CTA go through shared memory in a fixed order.
// The logits never go back to memory unless the caller asks for them.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2..5 epilogue.  Every wait is bounded.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "gemm_tc.cuh"
#include "ptx_sm100.cuh"
#include "route.cuh"

namespace moe {

template <int EPAD, int STAGES>
struct RouteTcSmem {
  static constexpr int BM = 128, BK = 64;
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = EPAD * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = EPAD < 32 ? 32 : EPAD;
  static constexpr int P_LD = EPAD + 1;   // row pitch of the softmax matrix (floats)
  static_assert(size_t(BM) * P_LD * 4 <= size_t(STAGES) * STAGE_BYTES,
                "the softmax matrix reuses the stage ring");
  struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    float lb[EPAD];
    float sb[EPAD];
    int amax[EPAD];
    float zq[4];
    int hist[4][kMaxExperts];
  };
  static constexpr size_t bytes() { return 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl); }
};

// Gates one token in registers.  l[e] holds the logits (+ logit bias) of
// experts e < E.  Writes the softmax into prow (shared, E entries), and returns
// the arg-max of the logits, the chosen experts, their weights and the
// log-sum-exp of the logits.
template <int EPAD, int KMAX>
__device__ __forceinline__ void gate_thread(float (&l)[EPAD], int E, int k, int route, int renorm,
                                            const float* sb, float* prow, int& amax,
                                            int (&sel)[KMAX], float (&wsel)[KMAX], float& lse) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  float m = NEG_INF;
  amax = 0;
  bool first = true;
#pragma unroll
  for (int e = 0; e < EPAD; ++e) {
    if (e < E) {
      float v = l[e];
      if (v != v) v = NEG_INF;   // NaN logits rank last
      l[e] = v;
      if (first || v > m) {
        m = v;
        amax = e;
        first = false;
      }
    }
  }
  float p[EPAD];
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < EPAD; ++e) {
    p[e] = (e < E) ? expf(l[e] - m) : 0.f;
    s += p[e];
  }
  lse = m + logf(s);
  const float inv_s = 1.0f / s;
#pragma unroll
  for (int e = 0; e < EPAD; ++e) {
    p[e] = p[e] * inv_s;
    if (e < E) prow[e] = p[e];
  }
  float bv[KMAX], sv[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    bv[j] = NEG_INF;
    sv[j] = 0.f;
    sel[j] = -1;
  }
#pragma unroll
  for (int e = 0; e < EPAD; ++e) {
    if (e < E) {
      float sc = (route == ROUTE_TOPK_SOFTMAX) ? l[e]
                 : (route == ROUTE_BIASED_SOFTMAX) ? p[e] + sb[e]
                                                   : p[e];
      if (sc != sc) sc = NEG_INF;
      // insertion: an empty slot or a strictly larger score takes the place
      float v = sc;
      float val = (route == ROUTE_TOPK_SOFTMAX) ? l[e] : p[e];
      int ix = e;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && (sel[j] < 0 || (ix >= 0 && v > bv[j]))) {
          const float tv = bv[j], tval = sv[j];
          const int ti = sel[j];
          bv[j] = v;
          sv[j] = val;
          sel[j] = ix;
          v = tv;
          val = tval;
          ix = ti;
        }
      }
    }
  }
  if (route == ROUTE_TOPK_SOFTMAX) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      wsel[j] = (j < k) ? expf(sv[j] - sv[0]) : 0.f;
      sum += wsel[j];
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) wsel[j] = wsel[j] / sum;
  } else if (route == ROUTE_BIASED_SOFTMAX || renorm) {
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) sum += (j < k) ? sv[j] : 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) wsel[j] = sv[j] / sum;
  } else {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) wsel[j] = sv[j];
  }
}

template <int EPAD, int KMAX, int STAGES>
__global__ void __launch_bounds__(192, 1)
k_route_tc(const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mW,
           const RouteArgs a) {
  using L = RouteTcSmem<EPAD, STAGES>;
  constexpr int BM = L::BM, BK = L::BK;
  static_assert(EPAD == 16 || EPAD == 32 || EPAD == 64, "expert tile");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  auto& c = *reinterpret_cast<typename L::Ctrl*>(smem + STAGES * L::STAGE_BYTES);
  float* sP = reinterpret_cast<float*>(smem);   // [128][P_LD] once the MMAs are done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  const int KB = (a.d + BK - 1) / BK;
  const int m0 = blockIdx.x * BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    mbar_init(&c.tfull, 1);
    mbar_init(&c.drain, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mX);
    tma_prefetch_desc(&mW);
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, L::TMEM_COLS);
    tmem_relinquish();
  }
  griddep_wait();
  griddep_launch_dependents();
  for (int e = threadIdx.x; e < EPAD; e += blockDim.x) {
    c.lb[e] = (a.logit_bias && e < E) ? a.logit_bias[e] : 0.f;
    c.sb[e] = (a.select_bias && e < E) ? a.select_bias[e] : 0.f;
    c.amax[e] = 0;
  }
  if (threadIdx.x < 4) c.zq[threadIdx.x] = 0.f;
  for (int i = threadIdx.x; i < 4 * kMaxExperts; i += blockDim.x) (&c.hist[0][0])[i] = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  volatile int* abort_flag = &c.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) armed[s] = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(&c.empty[stage], phase ^ 1u, abort_flag, a.dp.err,
                               DEV_ERR_WAIT_PRODUCER, kWaitLimitNs)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c.full[stage], L::STAGE_BYTES);
        tma_load_2d(sA + stage * L::A_BYTES, &mX, &c.full[stage], kb * BK, m0);
        tma_load_3d(sB + stage * L::B_BYTES, &mW, &c.full[stage], kb * BK, 0, 0);
#pragma unroll
        for (int s = 0; s < STAGES; ++s) armed[s] += (s == stage) ? 1u : 0u;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s)
          if (armed[s]) wait_timeout(&c.full[s], (armed[s] - 1u) & 1u, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, EPAD);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, issued = false;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_bounded(&c.full[stage], phase, abort_flag, a.dp.err, DEV_ERR_WAIT_MMA,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * L::A_BYTES);
        const uint32_t b0 = smem_u32(sB + stage * L::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16_f32(tmem_base, sdesc_kmajor_sw128(a0 + kk * 32),
                        sdesc_kmajor_sw128(b0 + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
        umma_commit(&c.empty[stage]);
        issued = true;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        umma_commit(&c.tfull);
      } else if (issued) {
        umma_commit(&c.drain);
        wait_timeout(&c.drain, 0, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ gating epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int t = m0 + row;
    const bool valid = t < a.T;
    int ok = 1;
    if (lane == 0)
      ok = mbar_wait_bounded(&c.tfull, 0, abort_flag, a.dp.err, DEV_ERR_WAIT_EPILOGUE,
                             kWaitLimitNs)
               ? 1
               : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      float l[EPAD];
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
      for (int cc = 0; cc < EPAD / 16; ++cc) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(trow + cc * 16, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int i = 0; i < 16; ++i) l[cc * 16 + i] = __uint_as_float(r[i]) + c.lb[cc * 16 + i];
      }
      if (valid && a.logits_out) {
#pragma unroll
        for (int e = 0; e < EPAD; ++e)
          if (e < E) a.logits_out[static_cast<int64_t>(t) * E + e] = l[e];
      }
      int amax;
      int sel[KMAX];
      float wsel[KMAX];
      float lse;
      float* prow = sP + row * L::P_LD;
      gate_thread<EPAD, KMAX>(l, E, a.k, a.route, a.renorm, c.sb, prow, amax, sel, wsel, lse);
      // z-loss term of this warp's tokens, a fixed shuffle tree
      float zz = valid ? lse * lse : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
      if (lane == 0) c.zq[q] = zz;
      if (!valid) {
#pragma unroll
        for (int e = 0; e < EPAD; ++e)
          if (e < E) prow[e] = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) sel[j] = -1;
      } else {
        atomicAdd(&c.amax[amax], 1);
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j < a.k) {
            a.idx[static_cast<int64_t>(t) * a.k + j] = sel[j];
            a.w[static_cast<int64_t>(t) * a.k + j] = wsel[j];
          }
        }
      }
      // this warp's 32 tokens are one ranking chunk
      if (m0 + q * 32 < a.T) rank_chunk_experts<KMAX>(a.dp, sel, (m0 >> 5) + q, c.hist[q]);
    }
    // the four epilogue warps: softmax column sums in row order, arg-max counts
    asm volatile("bar.sync 1, 128;" ::: "memory");
    // column e of the softmax matrix is summed by TPC = 128 / EPAD adjacent
    // threads (rows part, part + TPC, ...), then a fixed shuffle tree
    constexpr int TPC = BM / EPAD;
    const int eth = threadIdx.x - 64;
    const int ecol = eth / TPC, part = eth % TPC;
    float ps = 0.f;
    if (ok && ecol < E)
      for (int r2 = part; r2 < BM; r2 += TPC) ps += sP[r2 * L::P_LD + ecol];
#pragma unroll
    for (int o = 1; o < TPC; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    if (ok && ecol < E && part == 0) {
      if (ps != 0.f) atomicAdd(a.p_part + static_cast<int64_t>(ecol) * gridDim.x + blockIdx.x, ps);
      if (c.amax[ecol]) atomicAdd(a.a_tot + ecol, static_cast<unsigned int>(c.amax[ecol]));
    }
    if (ok && eth == 0) {   // z-loss row: the four warps in order
      const float zs = ((c.zq[0] + c.zq[1]) + c.zq[2]) + c.zq[3];
      if (zs != 0.f) atomicAdd(a.p_part + static_cast<int64_t>(E) * gridDim.x + blockIdx.x, zs);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
  if (arrive_last_block(a.dp.done)) {
    __shared__ int s_cnt[kMaxExperts];
    dispatch_finalize(a.dp, s_cnt);
    if (threadIdx.x == 0) *a.dp.done = 0u;
  }
}

}  // namespace moe
