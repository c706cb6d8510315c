// Block-scaled MX FP8 grouped GEMM on CTA pairs with 256 x 256 tiles: the
// compute-bound expert projections of layers whose experts hold many rows.
//
// Why a kernel of its own: an e4m3 MMA does twice the work of a bf16 one per
// byte of operand, so a tile must feed the tensor pipe twice as many bytes per
// cycle for the same arithmetic intensity.  256 x 128 pair tiles (the shape the
// bf16 pair kernel's tensor-memory budget leaves for MX scales) kept the pipe
// about 30 % busy on B300: the eight stages in flight could not cover the
// latency of 25 KB per 256 MMA cycles.  A 256 x 256 tile loads 36.5 KB per 512
// MMA cycles a CTA (32 KB of operands), and one N = 256 MMA per 32-K slice
// replaces two N = 128 ones (19 % less time for the Mixtral-shaped layer,
// measured on B300).  Its 256 accumulator columns leave no room for a second
// accumulator beside the scale ring, so the accumulator is single-buffered and
// the epilogue releases it as soon as it has copied it into registers.
//
// Layout of one stage (per CTA, the same offsets in both CTAs):
//   SFB the scale blocks of the tile's weight rows 0..127 and 128..255 (512
//       bytes each, the layout of mxfp8.cuh), each four times in a row:
//       [b0 b0 b0 b0 | b1 b1 b1 b1], 4 KB -- the packed weights' tile record
//       of the (expert, 128-K stage, 256-row tile), one TMA copy;
//   SFA the scale block of the CTA's 128 A rows, 512 bytes;
//   A   128 rows x 128 e4m3 bytes: rows 128 r .. 128 r + 127 of the pair tile
//       (CTA rank r);
//   B   128 weight rows x 128 bytes: rows 128 r .. 128 r + 127 of the tile.
// The scale stages come first, so that every descriptor of them, however its
// strides were read, stays inside the block's shared memory.
//
// The MMA thread of the even CTA issues one 256 x 256 x 32 block-scaled pair
// MMA per 32-K slice.  Its B scales fill 8 tensor-memory columns (column
// base + n / 32, lane n % 32 of every lane quarter); a single
// tcgen05.cp.128x256b writes all 8 at an 8-column aligned address from the
// replicated blocks (lane L receives 16 bytes of b0 and 16 of b1, both row
// L % 32), and a tcgen05.cp.32x128b.warpx4 writes the 4 columns of A scales.
// Both copies go from each CTA's shared memory into its own tensor memory
// (cta_group::2).  Copying b1 separately would take an address 4 columns
// off the 8-column grid, which this kernel avoids.  The records cost 4 KB of
// L2 reads a stage instead of 1 KB, but one TMA copy instead of eight: on
// B300 the copies a stage issues, more than its bytes, set the pace (one
// 4 KB copy ran the Mixtral-shaped layer 23 % faster than eight 512-byte ones
// and 11 % faster than two).
//
// Warps (320 threads): 0 producer (both CTAs), 1 tensor-memory allocation
// and, in the even CTA, the MMA issuer, 2..9 epilogue: warp w reads lane
// quarter w % 4 and column half (w - 2) / 4, i.e. one row and 128 columns a
// thread, loads all of them, arrives on the even CTA's `tempty` (16 arrivals
// free the accumulator for the next tile) and only then applies the
// activation, quantises or converts, and stores.
//
// Every wait is bounded as in gemm_tc2.cuh: a wait that runs out records
// MOE_DEV_ERR_* in the status word and raises the CTA's abort flag, and both
// CTAs still meet at the final cluster barrier.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "groups.cuh"
#include "ptx_sm100.cuh"

namespace moe {

// The block-scaled pair MMA (kind::mxf8f6f4, one E8M0 scale per 32 K): scale
// columns at the same tensor-memory addresses in both CTAs.
__device__ __forceinline__ void umma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// 128 rows x 32 bytes of shared memory into lanes 0..127, tensor-memory
// columns [taddr, taddr + 8) of each CTA of the pair (from that CTA's shared
// memory, the same offset).
__device__ __forceinline__ void tmem_cp_128x256b_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Descriptor of the replicated B scale blocks: 8-row x 16-byte core matrices,
// 128 bytes apart down the rows and 2048 bytes apart across the two 16-byte
// halves of a row (no swizzle).
__device__ __forceinline__ uint64_t sdesc_sfb_rep(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(2048 >> 4) << 16;            // leading byte offset: next 16 bytes
  d |= static_cast<uint64_t>(128 >> 4) << 32;             // stride byte offset: next 8 rows
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  return d;
}
// 32 rows x 16 bytes of shared memory into tensor-memory columns
// [taddr, taddr + 4) of each CTA of the pair (from that CTA's shared memory,
// the same offset), the rows copied into all four lane quarters.
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

template <int STAGES>
struct Mx2Smem {
  static constexpr int BM = 256, BN = 256, BK = 128;      // pair tile; K bytes a stage
  static constexpr uint32_t A_BYTES = 128 * 128;
  static constexpr uint32_t B_BYTES = 128 * 128;
  static constexpr uint32_t SFB_BYTES = 8 * 512;           // two blocks, four copies each
  static constexpr uint32_t SF_BYTES = SFB_BYTES + 512;    // + the A block
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SF_COL = 256;                  // scale ring after the accumulator
  static constexpr uint32_t SF_STRIDE = 16;                // SFA +0 (4 columns), SFB +8 (8)
  static_assert(SF_COL + STAGES * SF_STRIDE <= TMEM_COLS, "scale ring fits tensor memory");
  static_assert((STAGES * SF_BYTES) % 1024 == 0, "A and B stages 1024-byte aligned");
  struct Ctrl {
    uint64_t full[STAGES];    // even CTA: both CTAs' stage bytes landed
    uint64_t empty[STAGES];   // both CTAs: the stage's MMAs are done
    uint64_t tfull;           // both CTAs: accumulator ready
    uint64_t tempty;          // even CTA: all 16 epilogue warps copied it out
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    GroupTable tb;
  };
  static constexpr size_t bytes() { return 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl); }
  static_assert(1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl) <= 232448,
                "within the opt-in shared memory of a block");
};

// Activation and quantisation of one row's 128 accumulator columns held in
// registers (column half h of a 256-wide tile): writes the e4m3 codes and the
// row's scale bytes of the MX output.  GLU rows hold 64 gate columns then the
// 64 matching up columns (the packed weights' order) and give 64 outputs.
template <int EPI>
__device__ __forceinline__ void mx2_store_mx(const uint32_t (&a)[8][16], int col0, bool valid,
                                             int64_t orow, const __nv_bfloat16* bias,
                                             const TcArgs& args) {
  constexpr bool GLU = epi_glu(EPI);
  constexpr int NB = GLU ? 2 : 4;   // 32-column output blocks
  if (!valid) return;
  uint32_t sfw = 0;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 32 * b + i;
      float x = __uint_as_float(a[c >> 4][c & 15]);
      if (bias) x += __bfloat162float(bias[col0 + c]);
      if constexpr (GLU) {
        float u = __uint_as_float(a[(c + 64) >> 4][(c + 64) & 15]);
        if (bias) u += __bfloat162float(bias[args.N + col0 + c]);
        x = silu(x) * u;
      } else if (EPI == EPI_SILU_MX) {
        x = silu(x);
      } else {
        x = gelu_erf_as(x);
      }
      v[i] = x;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float inv;
    const uint32_t sbyte = mx_scale(amax, inv);
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      pk[i] = static_cast<uint32_t>(cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv)) |
              (static_cast<uint32_t>(cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv)) << 16);
    uint8_t* o = static_cast<uint8_t*>(args.out) + orow * args.ldo + col0 + 32 * b;
    *reinterpret_cast<uint4*>(o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4*>(o + 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    sfw |= sbyte << (8 * b);
  }
  uint8_t* sfp = args.sf_out + ((static_cast<int64_t>(col0 >> 7) * args.sf_out_rb + (orow >> 7)) * 512) +
                 (orow & 31) * 16 + ((orow & 127) >> 5) * 4;
  if constexpr (GLU) {
    *reinterpret_cast<uint16_t*>(sfp + ((col0 >> 5) & 3)) = static_cast<uint16_t>(sfw);
  } else {
    *reinterpret_cast<uint32_t*>(sfp) = sfw;
  }
}

// bf16 / fp32 outputs of one row's 128 accumulator columns (bias, the top-1
// gate weight of the fused combine).
template <int EPI>
__device__ __forceinline__ void mx2_store_dense(const uint32_t (&a)[8][16], int col0, bool valid,
                                                int64_t orow, float gate_w,
                                                const __nv_bfloat16* bias, const TcArgs& args) {
  if (!valid) return;
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const int col = col0 + 16 * cc;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(a[cc][i]);
    if (bias) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += __bfloat162float(bias[col + i]);
    }
    if constexpr (EPI == EPI_F32) {
      float* o = static_cast<float*>(args.out) + orow * args.ldo + col;
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
      if constexpr (EPI == EPI_SCATTER_BF16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= gate_w;
      }
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        pk[i] = *reinterpret_cast<uint32_t*>(&h);
      }
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + col;
      *reinterpret_cast<uint4*>(o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(o + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
}

// mA / mB: e4m3 codes of A (rows x K, 128 x 128 boxes) and of the weights
// ([groups, N, K], 128-row boxes); mSA: A's scale blocks (2 rows of 256
// bytes a block); mSB: the weights' 4 KB tile records (16 rows of 256 bytes).  Routed
// groups only (no shared experts); N (weight rows) a multiple of 256.
template <int STAGES, int EPI>
__global__ void __launch_bounds__(320, 1)
k_gemm_mx2(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mSA,
           const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mSB,
           const TcArgs args) {
  using L = Mx2Smem<STAGES>;
  constexpr int BM = L::BM, BK = L::BK;
  constexpr bool GLU = epi_glu(EPI);
  constexpr bool MXO = epi_mx_out(EPI);
  constexpr int BNO = GLU ? 128 : 256;   // output columns of a tile
  static_assert(!GLU || MXO, "GLU tiles quantise their output");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sSF = smem;
  uint8_t* sA = smem + STAGES * L::SF_BYTES;
  uint8_t* sB = sA + STAGES * L::A_BYTES;
  auto& c = *reinterpret_cast<typename L::Ctrl*>(smem + STAGES * L::STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: issues the MMAs
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const GroupSpec& gs = args.gs;
  const int G = gs.E;
  const int n_tiles = args.N / BNO;
  const int KB = args.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    mbar_init(&c.tfull, 1);
    mbar_init(&c.tempty, 16);
    mbar_init(&c.drain, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB);
    tma_prefetch_desc(&mSA);
    tma_prefetch_desc(&mSB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&c.tmem_base, L::TMEM_COLS);
    tmem_relinquish_pair();
  }
  griddep_wait();
  griddep_launch_dependents();
  build_group_table<BM>(gs, n_tiles, c.tb);
  if (args.pad_rows) pad_group_rows(c.tb, gs.E, args.pad_rows);
  tc_fence_before();
  cluster_sync_all();
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
        const int bz = gs.offsets ? g : 0;
        const int arow = c.tb.a_row0[g] + m_blk * BM + static_cast<int>(rank) * 128;
        const int brow = n_blk * 256 + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&c.empty[stage], phase ^ 1u, abort_flag, args.err,
                                 DEV_ERR_WAIT_PRODUCER, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
          if (rank == 0) mbar_arrive_expect_tx(&c.full[stage], 2 * L::STAGE_BYTES);
          uint8_t* sf = sSF + stage * L::SF_BYTES;
          tma_load_2d_pair(sA + stage * L::A_BYTES, &mA, fb, kb * BK, arow);
          tma_load_3d_pair(sB + stage * L::B_BYTES, &mB, fb, kb * BK, brow, bz);
          // the tile record of (expert, k stage, n tile): sfb_nb / 2 records a stage
          tma_load_2d_pair(sf, &mSB, fb, 0, 16 * ((bz * KB + kb) * (args.sfb_nb >> 1) + n_blk));
          tma_load_2d_pair(sf + L::SFB_BYTES, &mSA, fb, 0,
                           static_cast<int>(2 * (static_cast<int64_t>(kb) * args.sfa_rb + arow / 128)));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int t = pair; ok && t < total; t += n_pairs) {
        if (!mbar_wait_bounded(&c.tempty, acc_phase ^ 1u, abort_flag, args.err, DEV_ERR_WAIT_MMA,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&c.full[stage], phase, abort_flag, args.err, DEV_ERR_WAIT_MMA,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * L::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * L::B_BYTES);
          const uint32_t sf = smem_u32(sSF + stage * L::SF_BYTES);
          const uint32_t tsf = tmem_base + L::SF_COL + L::SF_STRIDE * static_cast<uint32_t>(stage);
          tmem_cp_32x128b_x4_pair(tsf, sdesc_sf_32x16(sf + L::SFB_BYTES));
          tmem_cp_128x256b_pair(tsf + 8, sdesc_sfb_rep(sf));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_mxf8_pair(tmem_base, sdesc_kmajor_sw128(a0 + kk * 32),
                           sdesc_kmajor_sw128(b0 + kk * 32), idesc_mxf8(BM, 256, kk, kk), tsf,
                           tsf + 8, (kb > 0 || kk != 0) ? 1u : 0u);
          umma_commit_pair(&c.empty[stage]);
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&c.tfull);
        acc_phase ^= 1u;
      }
      if (!ok) {
        // wait (bounded) for the MMAs in flight, then for the loads both CTAs
        // may still have in flight into the stages not yet seen full
        if (issued) {
          umma_commit_pair(&c.drain);
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
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3, h = (warp - 2) >> 2;
    const uint32_t tempty0 = map_to_cta(smem_u32(&c.tempty), 0);
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += n_pairs) {
      int g, m_blk, n_blk;
      decode_tile<BM>(c.tb, G, t, g, m_blk, n_blk);
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(&c.tfull, acc_phase, abort_flag, args.err, DEV_ERR_WAIT_EPILOGUE,
                               kWaitLimitNs)
                 ? 1
                 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      acc_phase ^= 1u;
      tc_fence_after();
      const uint32_t trow =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(128 * h);
      uint32_t a[8][16];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) tmem_ld_32x32b_x16(trow + 16 * cc, a[cc]);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) tmem_wait_ld(a[cc]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0);   // the accumulator is free

      const int row = q * 32 + lane;
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
      if (args.bias0) {
        const int64_t bstride = GLU ? 2 * static_cast<int64_t>(args.N) : args.N;
        bias = args.bias0 + static_cast<int64_t>(gs.offsets ? g : 0) * bstride;
      }
      const int col0 = n_blk * BNO + h * (BNO / 2);
      if constexpr (MXO)
        mx2_store_mx<EPI>(a, col0, valid, orow, bias, args);
      else
        mx2_store_dense<EPI>(a, col0, valid, orow, gate_w, bias, args);
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
