// MX FP8 operands of the expert GEMMs: e4m3 codes with one E8M0 scale per 32
// consecutive elements along K (the OCP Microscaling form), in the layout the
// block-scaled tcgen05 GEMM reads (gemm_tc.cuh, MX = true).
//
// Scale layout.  The scales of a [rows, K] operand are stored in 512-byte
// blocks, one per (128-column stage s = k / 128, 128-row block rb):
//   block (s, rb) at ((s * RB + rb) * 512) for activations (RB row blocks),
//   at (((g * KS + s) * NB + rb) * 512) for the weights of expert g,
// and inside a block the scale of row r = 128 rb + 32 c + i for k-block
// j = (k / 32) % 4 is byte 16 i + 4 c + j.  That is the order in which the MMA
// thread copies a block into tensor memory (32 lanes x 16 bytes, replicated
// into the four lane quarters).
//
//  k_quant_weights_mx  bf16 expert weights [G, N, K] -> packed codes + scales
//                      (SwiGLU weights: gate and up rows interleaved in
//                      64-row halves, so a 128-row tile holds 64 of each)
//  k_quant_rows_mx     expert-ordered bf16 rows (moe_grouped_ffn's x_perm)
//                      -> codes + scales at kPadRows-aligned group offsets
// The whole-layer pass quantises its rows in the permute kernel instead
// (dispatch.cuh, k_permute with MX output).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "groups.cuh"
#include "ptx_sm100.cuh"

namespace moe {

// Byte offset of the scale of (row r, k-block kb) inside an operand's scale
// blocks, given the block index base (s * RB for activations).
__host__ __device__ __forceinline__ int64_t mx_sf_offset(int64_t block, int r) {
  return block * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
}

// Quantises 8 consecutive bf16 values held by this lane, where lanes 4q..4q+3
// of the warp hold one 32-element block: returns the 8 codes, and the block's
// scale byte (the same in the four lanes).
__device__ __forceinline__ uint2 mx_quant8(const uint4 v, uint32_t& sbyte) {
  float f[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  float inv;
  sbyte = mx_scale(amax, inv);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = cvt_e4m3x2(f[2 * i] * inv, f[2 * i + 1] * inv);
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// Packed row p of a SwiGLU weight ([2F, K], gate rows then up rows) comes from
// gate row 64 t + i (p = 128 t + i, i < 64) or up row F + 64 t + i - 64.
__device__ __forceinline__ int glu_source_row(int p, int F) {
  const int t = p >> 7, i = p & 127;
  return i < 64 ? 64 * t + i : F + 64 * t + (i - 64);
}

// One warp per packed row of one expert: 256 elements a pass (8 a lane).
__global__ void __launch_bounds__(256)
k_quant_weights_mx(const __nv_bfloat16* __restrict__ w, int G, int N, int K, int glu,
                   uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nrows = static_cast<int64_t>(G) * N;
  if (gw >= nrows) return;
  const int g = static_cast<int>(gw / N), p = static_cast<int>(gw % N);
  const int src = glu ? glu_source_row(p, N / 2) : p;
  const __nv_bfloat16* row = w + (static_cast<int64_t>(g) * N + src) * K;
  uint8_t* out = codes + (static_cast<int64_t>(g) * N + p) * K;
  const int KS = K / 128, NB = N / 128;
  for (int k0 = 0; k0 < K; k0 += 256) {
    const int k = k0 + lane * 8;   // K % 128 == 0, so a pass holds whole blocks
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (k < K) v = __ldg(reinterpret_cast<const uint4*>(row + k));
    uint32_t sbyte;
    const uint2 q = mx_quant8(v, sbyte);
    if (k < K) {
      *reinterpret_cast<uint2*>(out + k) = q;
      if ((lane & 3) == 0) {
        const int kb = k >> 5;
        const int64_t blk = (static_cast<int64_t>(g) * KS + (kb >> 2)) * NB + (p >> 7);
        sf[mx_sf_offset(blk, p) + (kb & 3)] = static_cast<uint8_t>(sbyte);
      }
    }
  }
}

// Scale tile records of packed weights: for each (expert g, 128-K stage s,
// 256-row tile t) 4 KB at ((g * KS + s) * NT + t) * 4096 holding blocks 2t and
// 2t + 1 of the scale blocks, each four times: [b2t x4 | b2t+1 x4] (zeros for
// a block past the last, N / 128 odd).  One thread a 16-byte row of a copy.
__global__ void __launch_bounds__(256)
k_sf_tiles_mx(const uint8_t* __restrict__ sf, int64_t n_records, int NB, int NT,
              uint8_t* __restrict__ tiles) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_records * 256) return;
  const int64_t rec = i >> 8;                     // (g * KS + s) * NT + t
  const int chunk = static_cast<int>(i & 255);    // copy (chunk / 32), row (chunk % 32)
  const int t = static_cast<int>(rec % NT);
  const int64_t gs = rec / NT;                    // g * KS + s
  const int b = 2 * t + (chunk >> 7);
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (b < NB) v = *reinterpret_cast<const uint4*>(sf + (gs * NB + b) * 512 + (chunk & 31) * 16);
  *reinterpret_cast<uint4*>(tiles + i * 16) = v;
}

// Padded offsets of E groups: kPadRows * (blocks of kPadRows rows the groups
// before need), from the group starts `offsets` [E + 1] (or the kept counts
// when `kept` is given) -- the starts the GEMM derives (pad_group_rows).
// Every thread of the block must call it; warp 0 computes, the block syncs.
__device__ __forceinline__ void padded_offsets(const int32_t* offsets, const int32_t* kept,
                                               int E, int* s_poff) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int n = 0;
      if (e < E) n = kept ? __ldg(kept + e) : __ldg(offsets + e + 1) - __ldg(offsets + e);
      int v = (n + kPadRows - 1) / kPadRows;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (e < E) s_poff[e + 1] = (carry + v) * kPadRows;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_poff[0] = 0;
  }
  __syncthreads();
}

// Expert-ordered bf16 rows [offsets[E], K] -> codes [padded rows, K] and their
// scale blocks (RB row blocks), one warp per row.
__global__ void __launch_bounds__(256)
k_quant_rows_mx(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ offsets,
                int E, int K, int64_t RB, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ sf) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_poff[kMaxExperts + 1];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = __ldg(offsets + e);
  padded_offsets(offsets, nullptr, E, s_poff);
  const int lane = threadIdx.x & 31;
  const int n_rows = s_off[E];
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows; r += nw) {
    int lo = 0, hi = E;   // group g with s_off[g] <= r < s_off[g + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= r) lo = mid; else hi = mid;
    }
    const int prow = s_poff[lo] + (r - s_off[lo]);
    const __nv_bfloat16* row = x + static_cast<int64_t>(r) * K;
    uint8_t* out = codes + static_cast<int64_t>(prow) * K;
    for (int k0 = 0; k0 < K; k0 += 256) {
      const int k = k0 + lane * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (k < K) v = __ldg(reinterpret_cast<const uint4*>(row + k));
      uint32_t sbyte;
      const uint2 q = mx_quant8(v, sbyte);
      if (k < K) {
        *reinterpret_cast<uint2*>(out + k) = q;
        if ((lane & 3) == 0) {
          const int kb = k >> 5;
          sf[mx_sf_offset(static_cast<int64_t>(kb >> 2) * RB + (prow >> 7), prow) + (kb & 3)] =
              static_cast<uint8_t>(sbyte);
        }
      }
    }
  }
}

}  // namespace moe
