// Dispatch and combine: the local form of the all-to-all "dispatch -> compute
// -> combine" of expert parallelism (第7章 §7.5), on one GPU.
//
//  k_rank     one block per expert: counts its assignments and gives each a
//             stable rank in ascending t*k + j (the token order SimpleMoELayer's
//             torch.where produces), plus kept = min(count, C).
//  k_permute  exclusive scan of kept -> offsets; per token: slot of each of its
//             k assignments (or -1 past the capacity), perm_token, and the row
//             gather x -> x_perm (x read once, written k times, 16-byte vectors).
//  k_combine  out[t] = sum_j w[t,j] * y[slot_of[t,j]] + sum_s y_shared[s,t],
//             a gather in fixed order (no atomics); y is fp32, the sum is fp32
//             and out is rounded once to its dtype.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "groups.cuh"
#include "route.cuh"

namespace moe {

__device__ __forceinline__ int block_excl_scan(int v, int& total) {
  __shared__ int s_w[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) s_w[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_w[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    s_w[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  total = s_w[nw - 1];
  const int before = warp > 0 ? s_w[warp - 1] : 0;
  __syncthreads();
  return before + inc - v;
}

__global__ void __launch_bounds__(1024)
k_rank(const int32_t* __restrict__ idx, int Tk, int C, int32_t* __restrict__ rank,
       int32_t* __restrict__ counts, int32_t* __restrict__ kept) {
  const int e = blockIdx.x;
  const int nt = blockDim.x;
  const int seg = (Tk + nt - 1) / nt;
  const int beg = min(static_cast<int>(threadIdx.x) * seg, Tk);
  const int end = min(beg + seg, Tk);
  int c = 0;
  for (int a = beg; a < end; ++a) c += (__ldg(idx + a) == e) ? 1 : 0;
  int total;
  int r = block_excl_scan(c, total);
  for (int a = beg; a < end; ++a)
    if (__ldg(idx + a) == e) rank[a] = r++;
  if (threadIdx.x == 0) {
    if (counts) counts[e] = total;
    kept[e] = total < C ? total : C;
  }
}

// offsets of the kept rows, computed by every block into shared memory
__device__ __forceinline__ void scan_kept(const int32_t* kept, int E, int* s_off) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int v = e < E ? kept[e] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (e < E) s_off[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_off[0] = 0;
  }
  __syncthreads();
}

template <int KMAX>
__global__ void __launch_bounds__(256)
k_permute(const int32_t* __restrict__ idx, const int32_t* __restrict__ rank,
          const int32_t* __restrict__ kept, int T, int k, int E, int row_bytes,
          const uint8_t* __restrict__ x, uint8_t* __restrict__ x_perm,
          int32_t* __restrict__ offsets_out, int32_t* __restrict__ perm_token,
          int32_t* __restrict__ slot_of) {
  __shared__ int s_off[kMaxExperts + 1];
  scan_kept(kept, E, s_off);
  if (blockIdx.x == 0 && offsets_out)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets_out[e] = s_off[e];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nvec = row_bytes / 16;
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += nw) {
    int slot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      slot[j] = -1;
      if (j < k) {
        const int64_t a = static_cast<int64_t>(t) * k + j;
        const int e = __ldg(idx + a);
        const int r = __ldg(rank + a);
        slot[j] = (r < s_off[e + 1] - s_off[e]) ? s_off[e] + r : -1;
        if (lane == j) {
          slot_of[a] = slot[j];
          if (slot[j] >= 0 && perm_token) perm_token[slot[j]] = t;
        }
      }
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * row_bytes);
    for (int c = lane; c < nvec; c += 32) {
      const uint4 v = __ldg(src + c);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k && slot[j] >= 0)
          reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(slot[j]) * row_bytes)[c] = v;
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

template <typename TE, int KMAX>
__global__ void __launch_bounds__(256)
k_combine(const float* __restrict__ y, const int32_t* __restrict__ slot_of,
          const float* __restrict__ w, const float* __restrict__ y_shared, int n_shared, int T,
          int k, int d, TE* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nchunk = d / 8;
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += nw) {
    int slot[KMAX];
    float wt[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      slot[j] = -1;
      wt[j] = 0.f;
      if (j < k) {
        slot[j] = __ldg(slot_of + static_cast<int64_t>(t) * k + j);
        wt[j] = __ldg(w + static_cast<int64_t>(t) * k + j);
      }
    }
    for (int c = lane; c < nchunk; c += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && slot[j] >= 0) {
          float v[8];
          load8(y + static_cast<int64_t>(slot[j]) * d + c * 8, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wt[j], v[i], acc[i]);
        }
      }
      for (int s = 0; s < n_shared; ++s) {
        float v[8];
        load8(y_shared + (static_cast<int64_t>(s) * T + t) * d + c * 8, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += v[i];
      }
      store8(out + static_cast<int64_t>(t) * d + c * 8, acc);
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
  int gelu;
};

__global__ void __launch_bounds__(256) k_gemm_simt_f32(const SimtArgs a) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ GroupTable tb;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
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
    const float* B = (routed ? a.B0 : a.B1) + static_cast<int64_t>(gi) * a.N * a.K;
    const float* bias = routed ? a.bias0 : a.bias1;
    if (bias) bias += static_cast<int64_t>(gi) * a.N;
    const int rows = tb.rows[g];
    const int m0 = m_blk * BM, n0 = n_blk * BN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < a.K; k0 += BK) {
      for (int i = tid; i < BK * BM; i += 256) {
        const int r = i / BK, kk = i % BK;
        const int gr = m0 + r, gk = k0 + kk;
        As[kk][r] = (gr < rows && gk < a.K)
                        ? A[(static_cast<int64_t>(tb.a_row0[g]) + gr) * a.lda + gk]
                        : 0.f;
      }
      for (int i = tid; i < BK * BN; i += 256) {
        const int n = i / BK, kk = i % BK;
        const int gn = n0 + n, gk = k0 + kk;
        Bs[kk][n] = (gn < a.N && gk < a.K) ? B[static_cast<int64_t>(gn) * a.K + gk] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          av[i] = As[kk][ty * 4 + i];
          bv[i] = Bs[kk][tx * 4 + i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
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
        float v = acc[i][j] + (bias ? bias[gn] : 0.f);
        if (a.gelu) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
        o[gn] = v;
      }
    }
  }
}

}  // namespace moe
