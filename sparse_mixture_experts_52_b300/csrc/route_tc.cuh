// Router GEMM on the tensor cores with the gating in its epilogue, for bf16
// layers with E <= 16 experts.
//
// Every 128-token tile goes to a cluster of S CTAs (S = 1, 2 or 4, chosen so
// that a short batch still covers the SMs): CTA r of the cluster multiplies
// the tile's x rows by the r-th slice of the model dimension,
// partial[128, 16] = x_tile[:, Kr] . W_g[Kr, :] accumulating in TMEM
// (tcgen05, TMA-fed ring, as in gemm_tc.cuh).  The slice of W_g stays in
// shared memory for the whole kernel: the epilogue warps read it from W_g
// [d, E] as the layer holds it and write it in the K-major 128-byte-swizzled
// layout the MMA reads (so no transposed copy of W_g is made per call).  CTAs
// r > 0 then push their partial logits into CTA 0's shared memory (distributed
// shared memory) and the cluster meets at a barrier; CTA 0 adds them in rank
// order, and every epilogue thread owns one token (its TMEM lane) and gates
// it in registers: softmax over the E logits, the arg-max, the top-k by
// insertion in ascending expert order (strict comparisons, so the lower index
// wins equal scores), and the gate weights of the routing form.  The four
// epilogue warps hold 32 consecutive tokens each: exactly one ranking chunk,
// ranked from the registers.  The softmax column sums of the tile go through
// shared memory in a fixed order.  The logits never go back to memory unless
// the caller asks for them.
//
// Warp roles (192 threads): warp 0 TMA producer of x, warp 1 TMEM owner and
// MMA issuer, warps 2..5 W_g slice, then epilogue.  Every wait is bounded.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "ptx_sm100.cuh"
#include "route.cuh"

namespace moe {

template <int S>
struct RouteTcSmem {
  static constexpr int EPAD = 16, BM = 128, BK = 64;
  // the ring takes what the W_g slice leaves, up to 8 stages (more measured no
  // faster on B300: the kernel's fixed costs, not the stream, dominate)
  static constexpr int kMaxStages = 8;
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t W_KBLOCK = EPAD * 128;       // one 64-wide K block of W_g^T
  static constexpr uint32_t RED_BYTES = BM * EPAD * 4;   // one CTA's partial logits
  static constexpr uint32_t TMEM_COLS = 32;
  static constexpr int P_LD = EPAD + 1;   // row pitch of the softmax matrix (floats)
  static_assert(size_t(BM) * P_LD * 4 <= A_BYTES, "the softmax matrix reuses the stage ring");
  struct Ctrl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
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
  // the ring (`stages` x 16 KB), the W_g slice (kbs K blocks), the partials
  // of ranks 1..S-1
  __host__ __device__ static size_t w_off(int stages) { return size_t(stages) * A_BYTES; }
  __host__ __device__ static size_t red_off(int kbs, int stages) {
    return w_off(stages) + size_t(kbs) * W_KBLOCK;
  }
  __host__ __device__ static size_t ctrl_off(int kbs, int stages) {
    return red_off(kbs, stages) + size_t(S - 1) * RED_BYTES;
  }
  __host__ __device__ static size_t bytes(int kbs, int stages) {
    return 1024 + ctrl_off(kbs, stages) + sizeof(Ctrl);
  }
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

// K blocks of the model dimension that cluster rank r multiplies: KB blocks
// split as evenly as whole blocks allow.
__host__ __device__ __forceinline__ void route_k_range(int KB, int S, int r, int& kb0, int& kb1) {
  kb0 = static_cast<int>(static_cast<int64_t>(KB) * r / S);
  kb1 = static_cast<int>(static_cast<int64_t>(KB) * (r + 1) / S);
}

template <int KMAX, int S>
__global__ void __launch_bounds__(192, 1)
k_route_tc(const __grid_constant__ CUtensorMap mX, const __nv_bfloat16* __restrict__ w_g,
           int w_vec, int stages, const RouteArgs a) {
  using L = RouteTcSmem<S>;
  const int STAGES = stages;   // 1 .. L::kMaxStages
  constexpr int EPAD = L::EPAD, BM = L::BM, BK = L::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int E = a.E;
  const int KB = (a.d + BK - 1) / BK;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  int kb0, kb1;
  route_k_range(KB, S, static_cast<int>(rank), kb0, kb1);
  const bool has_k = kb1 > kb0;   // the host keeps S <= K blocks; an empty slice adds zeros
  const int kbs_max = (KB + S - 1) / S;
  uint8_t* sA = smem;
  uint8_t* sW = smem + L::w_off(STAGES);
  float* red = reinterpret_cast<float*>(smem + L::red_off(kbs_max, STAGES));
  auto& c = *reinterpret_cast<typename L::Ctrl*>(smem + L::ctrl_off(kbs_max, STAGES));
  float* sP = reinterpret_cast<float*>(smem);   // [128][P_LD] once the MMAs are done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / S, n_tiles = gridDim.x / S;
  const int m0 = tile * BM;

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
  if (warp == 0 && lane == 0) tma_prefetch_desc(&mX);
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
  bool epi_ok = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer of x
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;   // stage s has been armed issued / STAGES (+1 if s < issued % STAGES) times
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(&c.empty[stage], phase ^ 1u, abort_flag, a.dp.err,
                               DEV_ERR_WAIT_PRODUCER, kWaitLimitNs)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c.full[stage], L::A_BYTES);
        tma_load_2d(sA + stage * L::A_BYTES, &mX, &c.full[stage], kb * BK, m0);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        // wait (bounded) for the copies in flight: the last arming of each stage
        for (int s = 0; s < STAGES && s < issued; ++s) {
          const int armed = issued / STAGES + (s < issued % STAGES ? 1 : 0);
          wait_timeout(&c.full[s], static_cast<uint32_t>(armed - 1) & 1u, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    asm volatile("bar.sync 2, 160;" ::: "memory");   // the W_g slice is in place
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, EPAD);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, issued = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(&c.full[stage], phase, abort_flag, a.dp.err, DEV_ERR_WAIT_MMA,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * L::A_BYTES);
        const uint32_t b0 = smem_u32(sW + (kb - kb0) * L::W_KBLOCK);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16_f32(tmem_base, sdesc_kmajor_sw128(a0 + kk * 32),
                        sdesc_kmajor_sw128(b0 + kk * 32), idesc,
                        (kb > kb0 || kk != 0) ? 1u : 0u);
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
    // ------------------------------------------------------------ W_g slice
    // element (n, k) of W_g^T, K block j = (k - 64 kb0) / 64, at
    // j * 2048 + n * 128 + ((kk / 8) ^ (n % 8)) * 16 + (kk % 8) * 2, kk = k % 64:
    // 16-row x 128-byte tiles with the 128-byte swizzle TMA would have used
    const int eth = threadIdx.x - 64;
    const int k_lo = kb0 * BK, k_n = (kb1 - kb0) * BK;
    if (w_vec) {
      // E = 8 or 16 and W_g 16-byte aligned: a row of W_g is one or two
      // 16-byte loads; eight rows a thread in flight at once
      constexpr int RB = 8;
      for (int i0 = eth; i0 < k_n; i0 += 128 * RB) {
        uint32_t v[RB][8];
#pragma unroll
        for (int b = 0; b < RB; ++b) {
          const int i = i0 + 128 * b, k = k_lo + i;
          uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
          if (i < k_n && k < a.d) {
            const uint4* src = reinterpret_cast<const uint4*>(w_g + static_cast<int64_t>(k) * E);
            lo = __ldg(src);
            if (E == 16) hi = __ldg(src + 1);
          }
          v[b][0] = lo.x; v[b][1] = lo.y; v[b][2] = lo.z; v[b][3] = lo.w;
          v[b][4] = hi.x; v[b][5] = hi.y; v[b][6] = hi.z; v[b][7] = hi.w;
        }
#pragma unroll
        for (int b = 0; b < RB; ++b) {
          const int i = i0 + 128 * b;
          if (i < k_n) {
            const int j = i >> 6, kk = i & 63;
            uint8_t* col = sW + j * L::W_KBLOCK + (kk & 7) * 2;
#pragma unroll
            for (int n = 0; n < EPAD; ++n) {
              const uint16_t h = static_cast<uint16_t>(v[b][n >> 1] >> (16 * (n & 1)));
              *reinterpret_cast<uint16_t*>(col + n * 128 + (((kk >> 3) ^ (n & 7)) << 4)) =
                  n < E ? h : static_cast<uint16_t>(0);
            }
          }
        }
      }
    } else {
      for (int i = eth; i < k_n; i += 128) {
        const int k = k_lo + i;
        const int j = i >> 6, kk = i & 63;
        uint8_t* col = sW + j * L::W_KBLOCK + (kk & 7) * 2;
#pragma unroll
        for (int n = 0; n < EPAD; ++n) {
          __nv_bfloat16 v = __float2bfloat16_rn(0.f);
          if (n < E && k < a.d) v = w_g[static_cast<int64_t>(k) * E + n];
          *reinterpret_cast<__nv_bfloat16*>(col + n * 128 + (((kk >> 3) ^ (n & 7)) << 4)) = v;
        }
      }
    }
    fence_proxy_async_shared();   // read by the MMAs (async proxy)
    asm volatile("bar.sync 2, 160;" ::: "memory");
    int ok = 1;
    if (lane == 0)
      ok = mbar_wait_bounded(&c.tfull, 0, abort_flag, a.dp.err, DEV_ERR_WAIT_EPILOGUE,
                             kWaitLimitNs)
               ? 1
               : 0;
    epi_ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
    if constexpr (S > 1) {
      if (rank != 0) {
        // this rank's partial logits into CTA 0's shared memory, row-major
        const int q = warp & 3, row = q * 32 + lane;
        float v[EPAD];
        if (epi_ok && has_k) {
          tc_fence_after();
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16), r);
          tmem_wait_ld(r);
#pragma unroll
          for (int e = 0; e < EPAD; ++e) v[e] = __uint_as_float(r[e]);
        } else {
#pragma unroll
          for (int e = 0; e < EPAD; ++e) v[e] = 0.f;
        }
        const uint32_t dst = map_to_cta(
            smem_u32(red + (static_cast<size_t>(rank) - 1) * BM * EPAD + row * EPAD), 0);
#pragma unroll
        for (int e = 0; e < EPAD; e += 4)
          asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 4 * e),
                       "f"(v[e]), "f"(v[e + 1]), "f"(v[e + 2]), "f"(v[e + 3])
                       : "memory");
      }
    }
  }

  if constexpr (S > 1) {
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();   // the partials are in CTA 0 (release / acquire)
    tc_fence_after();
  }

  if (warp >= 2 && rank == 0) {
    // ------------------------------------------------------------ gating epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int t = m0 + row;
    const bool valid = t < a.T;
    const bool ok = epi_ok;
    if (ok) {
      float l[EPAD];
      uint32_t r[16];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16), r);
      tmem_wait_ld(r);
#pragma unroll
      for (int i = 0; i < EPAD; ++i) l[i] = has_k ? __uint_as_float(r[i]) : 0.f;
      // the other ranks' K slices, in rank order
#pragma unroll
      for (int rr = 1; rr < S; ++rr) {
        const float* pr = red + (rr - 1) * BM * EPAD + row * EPAD;
#pragma unroll
        for (int i = 0; i < EPAD; ++i) l[i] += pr[i];
      }
#pragma unroll
      for (int i = 0; i < EPAD; ++i) l[i] += c.lb[i];
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
      if (ps != 0.f) atomicAdd(a.p_part + static_cast<int64_t>(ecol) * n_tiles + tile, ps);
      if (c.amax[ecol]) atomicAdd(a.a_tot + ecol, static_cast<unsigned int>(c.amax[ecol]));
    }
    if (ok && eth == 0) {   // z-loss row: the four warps in order
      const float zs = ((c.zq[0] + c.zq[1]) + c.zq[2]) + c.zq[3];
      if (zs != 0.f) atomicAdd(a.p_part + static_cast<int64_t>(E) * n_tiles + tile, zs);
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
