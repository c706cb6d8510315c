// Dispatch and combine: the local form of the all-to-all "dispatch -> compute
// -> combine" of expert parallelism (第7章 §7.5), on one GPU.
//
//  k_permute  per token: the slot of each of its k assignments (or -1 past the
//             capacity) from the in-chunk ranks and per-chunk counts the
//             routing / ranking grid left (ascending t*k + j, the token order
//             SimpleMoELayer's torch.where produces), perm_token, and the row
//             gather x -> x_perm.
//  k_combine  out[t] = sum_j w[t,j] * y[slot_of[t,j]] + sum_s y_shared[s,t],
//             a gather in fixed order (no atomics); y is in the layer dtype,
//             the sum is fp32 and out is rounded once to its dtype.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "groups.cuh"
#include "mxfp8.cuh"
#include "route.cuh"

namespace moe {

// Slot of every assignment and the row gather.  Block b takes tokens
// [b*tpb, (b+1)*tpb) (tpb divides 32, so they lie in one chunk g).  Prologue:
// the block lists the distinct experts of its assignments and, for each,
// sums the counts of chunks 0..g-1 (hist row of that expert, 32 chunks = one
// 128-byte line per (expert, step) pair, spread over all threads, integer
// sums in shared memory).  Then one warp per token: the rank of assignment
// (t, j) inside its expert is that prefix plus its in-chunk rank; it is kept
// iff the rank is below kept[e], and lands in row offsets[e] + rank of
// x_perm.  x is read once and written k times with 16-byte vectors.  In a
// whole-layer pass of a top-1 layer without shared experts (whose combine is
// fused into the down-projection), tokens with no kept assignment get their
// zero output row here (zero_out), and one extra block reduces the routing
// statistics meanwhile.
//
// MXQ: the rows go out as MX FP8 for the block-scaled expert GEMM instead
// (bf16 rows, d a multiple of 128): each token's row is quantised once (32-
// element blocks over four lanes' 16-byte vectors) and its codes and scale
// bytes are written to the padded row of each kept slot: expert e's rows start
// at kPadRows * (row blocks of the experts before it), rank r inside.
template <int KMAX, bool MXQ = false>
__global__ void __launch_bounds__(256)
k_permute(const int32_t* __restrict__ idx, const int32_t* __restrict__ crank,
          const int32_t* __restrict__ hist, const int32_t* __restrict__ kept,
          const int32_t* __restrict__ offsets, int T, int k, int E, int ncs, int tpb,
          int row_bytes, const uint8_t* __restrict__ x, uint8_t* __restrict__ x_perm,
          int32_t* __restrict__ perm_token, int32_t* __restrict__ slot_of,
          uint8_t* __restrict__ zero_out, const StatsArgs st, uint8_t* __restrict__ xq_sf,
          int64_t sf_rb) {
  __shared__ int s_pre[kMaxExperts];
  __shared__ int s_list[32 * kMaxK];
  __shared__ unsigned int s_mark[kMaxExperts / 32];
  __shared__ int s_n;
  __shared__ int s_poff[MXQ ? kMaxExperts + 1 : 1];
  griddep_wait();
  griddep_launch_dependents();
  if (st.p_part) {   // the last stats_blocks(E, 8) blocks reduce the routing statistics
    const int nsb = stats_blocks(st.E, 8);
    const int sb = static_cast<int>(blockIdx.x) - (static_cast<int>(gridDim.x) - nsb);
    if (sb >= 0) {
      stats_reduce(st, sb, nsb);
      return;
    }
  }
  if constexpr (MXQ) padded_offsets(nullptr, kept, E, s_poff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * tpb, t1 = min(t0 + tpb, T);
  const int g = t0 / kChunk;
  if (tid < kMaxExperts / 32) s_mark[tid] = 0u;
  if (tid == 0) s_n = 0;
  __syncthreads();
  for (int a = t0 * k + tid; a < t1 * k; a += blockDim.x) {
    const int e = __ldg(idx + a);
    if (e >= 0 && e < E) {
      const unsigned int bit = 1u << (e & 31);
      if (!(atomicOr(&s_mark[e >> 5], bit) & bit)) {
        s_pre[e] = 0;
        s_list[atomicAdd(&s_n, 1)] = e;
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  const int steps = (g + 31) / 32;   // 32-chunk steps before chunk g
  for (int p = tid; p < n * steps; p += blockDim.x) {
    const int e = s_list[p / steps];
    const int c0 = (p % steps) * 32;
    const int4* src = reinterpret_cast<const int4*>(hist + static_cast<int64_t>(e) * ncs + c0);
    int4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(src + i);
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + 4 * i;
      sum += (c < g ? v[i].x : 0) + (c + 1 < g ? v[i].y : 0) + (c + 2 < g ? v[i].z : 0) +
             (c + 3 < g ? v[i].w : 0);
    }
    if (sum) atomicAdd(&s_pre[e], sum);
  }
  __syncthreads();
  const int nvec = row_bytes / 16;
  for (int t = t0 + warp; t < t1; t += blockDim.x >> 5) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * row_bytes);
    // the first vectors of the row are in flight while the slots resolve
    constexpr int PF = 4;
    uint4 v[PF];
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      const int c = lane + 32 * i;
      if (c < nvec) v[i] = __ldg(src + c);
    }
    // lane j < k resolves slot j; the warp then shares the k slots
    int my_slot = -1, my_prow = -1;
    // a token's expert indices, for the repeated-index check of the ranking
    const int my_e = lane < k ? __ldg(idx + static_cast<int64_t>(t) * k + lane) : -1;
    bool repeated = false;
#pragma unroll
    for (int jj = 0; jj < KMAX; ++jj) {
      const int o = __shfl_sync(0xffffffffu, my_e, jj);
      repeated |= (jj < k && jj < lane && o == my_e);
    }
    if (lane < k) {
      const int64_t a = static_cast<int64_t>(t) * k + lane;
      const int e = my_e;
      if (e >= 0 && e < E && !repeated) {
        const int r = s_pre[e] + __ldg(crank + a);
        my_slot = (r < __ldg(kept + e)) ? __ldg(offsets + e) + r : -1;
        if constexpr (MXQ) my_prow = my_slot >= 0 ? s_poff[e] + r : -1;
      }
      slot_of[a] = my_slot;
      if (my_slot >= 0 && perm_token) perm_token[my_slot] = t;
    }
    int slot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
    if (zero_out) {   // a token with every assignment dropped gets a zero output row
      bool any = false;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) any |= (j < k && slot[j] >= 0);
      if (!any) {
        uint4* o = reinterpret_cast<uint4*>(zero_out + static_cast<int64_t>(t) * row_bytes);
        for (int c = lane; c < nvec; c += 32) o[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if constexpr (MXQ) {
      int prow[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) prow[j] = __shfl_sync(0xffffffffu, my_prow, j);
      const int d = row_bytes / 2;   // bf16 elements; codes are one byte each
      for (int c0 = 0; c0 < nvec; c0 += 32 * PF) {
#pragma unroll
        for (int i = 0; i < PF; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c0 > 0) v[i] = c < nvec ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
          else if (c >= nvec) v[i] = make_uint4(0u, 0u, 0u, 0u);
          uint32_t sbyte;
          const uint2 q = mx_quant8(v[i], sbyte);   // every lane: the block takes 4 lanes
          if (c < nvec) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
              if (j < k && prow[j] >= 0) {
                *reinterpret_cast<uint2*>(x_perm + static_cast<int64_t>(prow[j]) * d + c * 8) = q;
                if ((lane & 3) == 0)   // k-block c / 4: stage c / 16, byte (c / 4) % 4
                  xq_sf[mx_sf_offset(static_cast<int64_t>(c >> 4) * sf_rb + (prow[j] >> 7),
                                     prow[j]) + ((c >> 2) & 3)] = static_cast<uint8_t>(sbyte);
              }
            }
          }
        }
      }
    } else {
    for (int c0 = 0; c0 < nvec; c0 += 32 * PF) {
      if (c0 > 0) {
#pragma unroll
        for (int i = 0; i < PF; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < nvec) v[i] = __ldg(src + c);
        }
      }
#pragma unroll
      for (int i = 0; i < PF; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < nvec) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if (j < k && slot[j] >= 0)
              reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(slot[j]) * row_bytes)[c] = v[i];
        }
      }
    }
    }
  }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Eight consecutive elements of a row kept as loaded (bf16 packed in one
// 16-byte vector), converted to fp32 only when they are summed.
template <typename TE>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    v = __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ void fma_into(float w, float (&acc)[8]) const {
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(w, __uint_as_float(h[i] << 16), acc[2 * i]);
      acc[2 * i + 1] = fmaf(w, __uint_as_float(h[i] & 0xffff0000u), acc[2 * i + 1]);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void fma_into(float w, float (&acc)[8]) const {
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, f[i], acc[i]);
  }
};

// out[t] = sum_j w[t,j] * y[slot_of[t,j]] + sum_s y_shared[s,t]: one warp per
// token, fp32 sums in ascending j then s, one rounding.  The expert outputs
// (TY) are in the layer dtype, or fp32 for a bf16 layer that keeps them so;
// out is in the layer dtype (TO).  The rows of up to
// eight slots (four for fp32; U 16-byte vectors per lane each, kept packed as
// loaded) are requested together before any is summed, so a warp has up to
// 8 * U * 512 bytes in flight; 64 registers a thread let every token of a
// 4096-token batch hold a warp at once.
template <typename TY, typename TO, int KMAX, int U>
__global__ void __launch_bounds__(256, 4)
k_combine(const TY* __restrict__ y, const int32_t* __restrict__ slot_of,
          const float* __restrict__ w, const TY* __restrict__ y_shared, int n_shared, int T,
          int k, int d, TO* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nchunk = d / 8;
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += nw) {
    // lane j < k holds slot j and its weight; the warp reads them by shuffle
    int my_slot = -1;
    float my_w = 0.f;
    if (lane < k) {
      my_slot = __ldg(slot_of + static_cast<int64_t>(t) * k + lane);
      my_w = __ldg(w + static_cast<int64_t>(t) * k + lane);
    }
    // slots whose rows are in flight together (fp32 vectors take twice the registers)
    constexpr int QMAX = sizeof(TY) == 2 ? 8 : 4;
    constexpr int Q = KMAX < QMAX ? KMAX : QMAX;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
#pragma unroll
      for (int j0 = 0; j0 < KMAX; j0 += Q) {
        Raw8<TY> v[Q][U];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const int s = __shfl_sync(0xffffffffu, my_slot, j0 + q);
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int c = c0 + lane + 32 * u;
            if (s >= 0 && c < nchunk) v[q][u].load(y + static_cast<int64_t>(s) * d + c * 8);
          }
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const int s = __shfl_sync(0xffffffffu, my_slot, j0 + q);
          const float wq = __shfl_sync(0xffffffffu, my_w, j0 + q);
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (s >= 0 && c0 + lane + 32 * u < nchunk) v[q][u].fma_into(wq, acc[u]);
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

// ---------------------------------------------------------------------------
// fp32 grouped GEMM on the CUDA cores (no TF32: its 10-bit mantissa would not
// meet a 1e-4 relative tolerance).  64 x 64 tiles, 256 threads, 4 x 4 each.
struct SimtArgs {
  GroupSpec gs;
  int N, K;
  const float* A0;
  const float* A1;
  int64_t lda;
  const float* B0;   // [E, N, K]
  const float* B1;   // [S, N, K]
  const float* bias0;
  const float* bias1;
  float* out;        // routed groups' rows
  float* out1;       // shared groups' rows
  int64_t ldo;
  int act;           // SIMT_ACT_*
};

// Epilogue of k_gemm_simt_f32.  SIMT_ACT_SWIGLU: B (and the bias) hold 2N
// rows, the gate projection's then the up projection's, and the output is
// SiLU(gate) * up over N columns.
enum : int { SIMT_ACT_NONE = 0, SIMT_ACT_GELU = 1, SIMT_ACT_SILU = 2, SIMT_ACT_SWIGLU = 3 };

__device__ __forceinline__ float simt_silu(float v) { return v / (1.0f + expf(-v)); }

template <bool GLU>
__global__ void __launch_bounds__(256) k_gemm_simt_f32(const SimtArgs a) {
  constexpr int BM = 64, BN = 64, BK = 16;
  constexpr int LA = BK * BM / 256, LB = BK * BN / 256;   // elements per thread per k-step
  constexpr int NB = GLU ? 2 : 1;                         // B tiles: gate (and up)
  griddep_wait();
  griddep_launch_dependents();
  __shared__ GroupTable tb;
  __shared__ float As[2][BK][BM + 4];
  __shared__ float Bs[2][NB][BK][BN + 4];
  const GroupSpec& gs = a.gs;
  const int G = gs.E + gs.n_shared;
  const int n_tiles = (a.N + BN - 1) / BN;
  build_group_table<BM>(gs, n_tiles, tb);
  const int total = tb.tile_start[G];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    int g, m_blk, n_blk;
    decode_tile<BM>(tb, G, t, g, m_blk, n_blk);
    const bool routed = g < gs.E;
    const float* A = (routed || gs.shared_a_sel == 0) ? a.A0 : a.A1;
    const int gi = routed ? (gs.offsets ? g : 0) : g - gs.E;
    const float* B = (routed ? a.B0 : a.B1) + static_cast<int64_t>(gi) * NB * a.N * a.K;
    const float* bias = routed ? a.bias0 : a.bias1;
    if (bias) bias += static_cast<int64_t>(gi) * NB * a.N;
    const int rows = tb.rows[g];
    const int m0 = m_blk * BM, n0 = n_blk * BN;
    const int64_t arow0 = tb.a_row0[g];
    // global -> registers for k-step k0 (the next step's loads are in flight
    // while the current step computes from shared memory)
    float ra[LA], rb[NB][LB];
    auto fetch = [&](int k0) {
#pragma unroll
      for (int q = 0; q < LA; ++q) {
        const int i = tid + 256 * q;
        const int r = i / BK, kk = i % BK;
        const int gr = m0 + r, gk = k0 + kk;
        ra[q] = (gr < rows && gk < a.K) ? __ldg(A + (arow0 + gr) * a.lda + gk) : 0.f;
      }
#pragma unroll
      for (int h = 0; h < NB; ++h)
#pragma unroll
        for (int q = 0; q < LB; ++q) {
          const int i = tid + 256 * q;
          const int n = i / BK, kk = i % BK;
          const int gn = n0 + n, gk = k0 + kk;
          rb[h][q] = (gn < a.N && gk < a.K)
                         ? __ldg(B + (static_cast<int64_t>(h) * a.N + gn) * a.K + gk)
                         : 0.f;
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
      for (int q = 0; q < LA; ++q) {
        const int i = tid + 256 * q;
        As[buf][i % BK][i / BK] = ra[q];
      }
#pragma unroll
      for (int h = 0; h < NB; ++h)
#pragma unroll
        for (int q = 0; q < LB; ++q) {
          const int i = tid + 256 * q;
          Bs[buf][h][i % BK][i / BK] = rb[h][q];
        }
    };
    float acc[NB][4][4] = {};
    fetch(0);
    stash(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < a.K; k0 += BK) {
      const bool more = k0 + BK < a.K;
      if (more) fetch(k0 + BK);
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float av[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[buf][kk][ty * 4 + i];
#pragma unroll
        for (int h = 0; h < NB; ++h) {
          float bv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) bv[j] = Bs[buf][h][kk][tx * 4 + j];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][i][j] = fmaf(av[i], bv[j], acc[h][i][j]);
        }
      }
      if (more) stash(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gr = m0 + ty * 4 + i;
      if (gr >= rows) continue;
      float* o = (routed ? a.out : a.out1) + (static_cast<int64_t>(tb.out_row0[g]) + gr) * a.ldo;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int gn = n0 + tx * 4 + j;
        if (gn >= a.N) continue;
        float v = acc[0][i][j] + (bias ? bias[gn] : 0.f);
        if (GLU) {
          const float up = acc[NB - 1][i][j] + (bias ? bias[a.N + gn] : 0.f);
          v = simt_silu(v) * up;
        } else if (a.act == SIMT_ACT_GELU) {
          v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
        } else if (a.act == SIMT_ACT_SILU) {
          v = simt_silu(v);
        }
        o[gn] = v;
      }
    }
  }
}

}  // namespace moe
