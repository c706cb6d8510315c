// Grouped GEMM on CTA pairs (tcgen05 cta_group::2): the same product as
// gemm_tc.cuh, for compute-bound layers whose experts hold many rows.
//
// Two CTAs of a cluster share one 256 x BN tile.  CTA rank r holds rows
// 128 r .. 128 r + 127 of the tile's A and columns r BN/2 .. (r + 1) BN/2 - 1
// of its B (B rows of the expert's weight) in shared memory, at the same
// offsets in both CTAs; the even CTA issues one 256 x BN x 16 MMA per k-step,
// which reads both CTAs' halves, and each CTA's tensor memory receives its
// own 128 rows of the fp32 accumulator.  Per SM a k-step then reads 16 KB of
// A and B instead of 24 KB for a 128 x 256 tile, and every weight slab that
// crosses L2 feeds 256 rows.
//
// Pipeline (per CTA, 192 threads): warp 0 lane 0 loads its halves of the
// stage with TMA and signals the even CTA's `full` barrier (the even CTA
// expects both halves' bytes); warp 1 lane 0 of the even CTA issues the MMAs
// and commits to the `empty` barriers of both CTAs (multicast), and, per
// tile, to both CTAs' `tfull`; warps 2..5 of each CTA read their rows from
// tensor memory, apply the epilogue and arrive on the even CTA's `tempty`
// (eight warps in all).  Tiles go round robin over the pairs: pair p takes
// tiles p, p + P, ... in the group-major order of groups.cuh with 256-row
// blocks.
//
// The block-scaled MX FP8 product runs on its own pair kernel (gemm_mx2.cuh).
//
// Every wait is bounded; a wait that runs out records MOE_DEV_ERR_* in the
// status word and raises the CTA's abort flag; both CTAs still meet at the
// final cluster barrier (their other waits give up in turn), so a bad launch
// cannot hang the GPU.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "gemm_tc.cuh"
#include "groups.cuh"
#include "ptx_sm100.cuh"

namespace moe {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `local` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// TMA 2-D / 3-D load into this CTA's shared memory, completing on an mbarrier
// that may live in the peer CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem of both CTAs] (+)= A[both CTAs' smem] * B[both CTAs' smem]^T, M = 256.
__device__ __forceinline__ void umma_bf16_f32_pair(uint32_t d_tmem, uint64_t a_desc,
                                                   uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` (same offset) in both CTAs of the pair when the pair
// MMAs issued so far by this thread are done.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

template <int BN, int STAGES>
struct Tc2Smem {
  static constexpr int BM = 256, BK = 64;                // tile rows (pair); K per stage
  static constexpr uint32_t A_BYTES = 128 * 128;         // this CTA's 128 rows
  static constexpr uint32_t B_BYTES = (BN / 2) * 128;    // this CTA's BN/2 columns
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;   // bytes of one CTA
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  struct Ctrl {
    uint64_t full[STAGES];    // even CTA: both halves landed
    uint64_t empty[STAGES];   // both CTAs: the stage's MMAs are done
    uint64_t tfull[2];        // both CTAs: accumulator ready
    uint64_t tempty[2];       // even CTA: both CTAs' epilogues read it
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    GroupTable tb;
  };
  static constexpr size_t bytes() {
    return 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl);
  }
};

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(192, 1)
k_gemm_tc2(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
           const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
           const TcArgs args) {
  using L = Tc2Smem<BN, STAGES>;
  constexpr int BM = L::BM, BK = L::BK;
  constexpr int NCC = BN / 16;
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 256");
  static_assert(!epi_mx_out(EPI), "MX outputs come from the MX pair kernel");
  constexpr bool GLU = epi_glu(EPI);
  constexpr int BNO = GLU ? BN / 2 : BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  auto& c = *reinterpret_cast<typename L::Ctrl*>(smem + STAGES * L::STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: issues the MMAs
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const GroupSpec& gs = args.gs;
  const int G = gs.E + gs.n_shared;
  const int n_tiles = (args.N + BNO - 1) / BNO;
  const int KB = (args.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c.tfull[a], 1);
      mbar_init(&c.tempty[a], 8);
    }
    mbar_init(&c.drain, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA0);
    tma_prefetch_desc(&mB0);
    if (gs.n_shared > 0) {
      tma_prefetch_desc(&mA1);
      tma_prefetch_desc(&mB1);
    }
  }
  if (warp == 1) {   // one warp of each CTA allocates the pair's tensor memory
    tmem_alloc_pair(&c.tmem_base, L::TMEM_COLS);
    tmem_relinquish_pair();
  }
  griddep_wait();
  griddep_launch_dependents();
  build_group_table<BM>(gs, n_tiles, c.tb);
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers are initialised before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int total = c.tb.tile_start[G];
  volatile int* abort_flag = &c.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint32_t full0 = map_to_cta(smem_u32(&c.full[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; ok && t < total; t += n_pairs) {
        int g, m_blk, n_blk;
        decode_tile<BM>(c.tb, G, t, g, m_blk, n_blk);
        const bool routed = g < gs.E;
        const CUtensorMap* ma = (routed || gs.shared_a_sel == 0) ? &mA0 : &mA1;
        const CUtensorMap* mb = routed ? &mB0 : &mB1;
        const int bz = routed ? (gs.offsets ? g : 0) : g - gs.E;
        const int arow = c.tb.a_row0[g] + m_blk * BM + static_cast<int>(rank) * 128;
        // B rows of this CTA's half: GLU tiles hold the gate rows (rank 0) and
        // the matching up rows (rank 1); others the two halves of BN rows
        const int brow = GLU ? static_cast<int>(rank) * args.N + n_blk * BNO
                             : n_blk * BN + static_cast<int>(rank) * (BN / 2);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&c.empty[stage], phase ^ 1u, abort_flag, args.err,
                                 DEV_ERR_WAIT_PRODUCER, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
          if (rank == 0) mbar_arrive_expect_tx(&c.full[stage], 2 * L::STAGE_BYTES);
          tma_load_2d_pair(sA + stage * L::A_BYTES, ma, fb, kb * BK, arow);
          tma_load_3d_pair(sB + stage * L::B_BYTES, mb, fb, kb * BK, brow, bz);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // after a give-up, loads already issued complete on the even CTA's
      // barriers; the final cluster barrier keeps this CTA's shared memory
      // alive until then (the even CTA drains them before it arrives)
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      int landed = 0;   // stages whose full phase this thread has seen
      for (int t = pair; ok && t < total; t += n_pairs) {
        if (!mbar_wait_bounded(&c.tempty[acc], acc_phase ^ 1u, abort_flag, args.err,
                               DEV_ERR_WAIT_MMA, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&c.full[stage], phase, abort_flag, args.err, DEV_ERR_WAIT_MMA,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          ++landed;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * L::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * L::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16_f32_pair(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32),
                               sdesc_kmajor_sw128(b0 + kk * 32), idesc,
                               (kb > 0 || kk != 0) ? 1u : 0u);
          umma_commit_pair(&c.empty[stage]);
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&c.tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        // wait (bounded) for the MMAs in flight, then for the loads both CTAs
        // may still have in flight into the stages not yet seen full
        if (issued) {
          umma_commit_pair(&c.drain);   // arrives on both CTAs' drain barriers
          wait_timeout(&c.drain, 0, kDrainLimitNs);
        }
        for (int i = 0; i < STAGES; ++i) {
          wait_timeout(&c.full[stage], phase, kDrainLimitNs);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      (void)landed;
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const uint32_t tempty0 = map_to_cta(smem_u32(&c.tempty[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += n_pairs) {
      int g, m_blk, n_blk;
      decode_tile<BM>(c.tb, G, t, g, m_blk, n_blk);
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(&c.tfull[acc], acc_phase, abort_flag, args.err,
                               DEV_ERR_WAIT_EPILOGUE, kWaitLimitNs)
                 ? 1
                 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(acc * BN);
      const int row = q * 32 + lane;
      const bool routed = g < gs.E;
      const int row_in_grp = m_blk * BM + static_cast<int>(rank) * 128 + row;
      const bool valid = row_in_grp < c.tb.rows[g];
      int64_t orow = static_cast<int64_t>(c.tb.out_row0[g]) + row_in_grp;
      float gate_w = 1.f;
      if (EPI == EPI_SCATTER_BF16 && valid) {
        const int tok = __ldg(args.scatter_token + orow);
        gate_w = __ldg(args.scatter_w + tok);
        orow = tok;
      }
      const __nv_bfloat16* bias = nullptr;
      {
        const int64_t bstride = GLU ? 2 * static_cast<int64_t>(args.N) : args.N;
        if (routed && args.bias0) bias = args.bias0 + static_cast<int64_t>(gs.offsets ? g : 0) * bstride;
        if (!routed && args.bias1) bias = args.bias1 + static_cast<int64_t>(g - gs.E) * bstride;
      }
      constexpr int NOUT = GLU ? NCC / 2 : NCC;
#pragma unroll 1
      for (int cc = 0; cc < NOUT; ++cc) {
        uint32_t r[16], ru[GLU ? 16 : 1];
        tmem_ld_32x32b_x16(trow + cc * 16, r);
        tmem_wait_ld(r);
        if constexpr (GLU) {
          tmem_ld_32x32b_x16(trow + (cc + NCC / 2) * 16, ru);
          tmem_wait_ld(ru);
        }
        const int col = n_blk * BNO + cc * 16;
        if (!valid || col >= args.N) continue;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
        if (bias) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (col + i < args.N) v[i] += __bfloat162float(bias[col + i]);
        }
        if (EPI == EPI_F32) {
          float* o = static_cast<float*>(routed ? args.out : args.out1) + orow * args.ldo + col;
          if (col + 16 <= args.N) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          } else {
            for (int i = 0; i < 16 && col + i < args.N; ++i) o[i] = v[i];
          }
          continue;
        }
        if constexpr (GLU) {
          float w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = __uint_as_float(ru[i]);
          if (bias) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (col + i < args.N) w[i] += __bfloat162float(bias[args.N + col + i]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = silu(v[i]) * w[i];
        } else if (EPI == EPI_SILU_BF16) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = silu(v[i]);
        } else if (EPI == EPI_GELU_BF16) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = gelu_erf(v[i]);
        } else if (EPI == EPI_SCATTER_BF16) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= gate_w;
        }
        __nv_bfloat16* o =
            static_cast<__nv_bfloat16*>(routed ? args.out : args.out1) + orow * args.ldo + col;
        if (col + 16 <= args.N) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            pk[i] = *reinterpret_cast<uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(o + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        } else {
          for (int i = 0; i < 16 && col + i < args.N; ++i) o[i] = __float2bfloat16_rn(v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  cluster_sync_all();   // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace moe
