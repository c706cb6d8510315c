// Group table of a grouped GEMM: which rows of the activation matrix belong
// to which expert, read on the device from the dispatch offsets so that the
// per-expert row counts never travel to the host.
#pragma once
#include <cstdint>

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxShared = 4;
constexpr int kMaxGroups = kMaxExperts + kMaxShared;

// Groups 0..E-1 are the routed experts: rows [offsets[g], offsets[g+1]) of A
// and of the output (or one dense group of `dense_rows` rows when offsets is
// null).  Groups E..E+n_shared-1 are the shared experts: `shared_rows` rows
// each.  Shared group s reads A rows from shared_a_row0 + s * shared_a_stride
// (stride 0 when every shared expert reads the same tokens, shared_rows when
// each has its own stacked hidden rows) and writes output rows from
// shared_out_row0 + s * shared_rows.
struct GroupSpec {
  const int32_t* offsets;
  int E;
  int dense_rows;
  int n_shared;
  int shared_rows;
  int shared_a_sel;     // A operand of shared groups: 0 = map/pointer 0, 1 = map/pointer 1
  int shared_a_row0;
  int shared_out_row0;
  int shared_a_stride;
};

struct GroupTable {
  int tile_start[kMaxGroups + 1];  // first tile of each group; [G] = total tiles
  int rows[kMaxGroups];
  int a_row0[kMaxGroups];
  int out_row0[kMaxGroups];
};

// Fills `tb` (shared memory) for tiles of BM rows x n_tiles column blocks,
// ordered group-major, then column block, then row block (row block fastest, so
// CTAs running at the same time share one weight slab).  Every thread of the
// block must call it (it synchronises the block).
template <int BM>
__device__ __forceinline__ void build_group_table(const GroupSpec& gs, int n_tiles,
                                                  GroupTable& tb) {
  const int G = gs.E + gs.n_shared;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int rows, arow, orow;
    if (g < gs.E) {
      if (gs.offsets) {
        const int b = gs.offsets[g], e = gs.offsets[g + 1];
        rows = e - b;
        arow = b;
        orow = b;
      } else {
        rows = gs.dense_rows;
        arow = 0;
        orow = 0;
      }
    } else {
      const int s = g - gs.E;
      rows = gs.shared_rows;
      arow = gs.shared_a_row0 + s * gs.shared_a_stride;
      orow = gs.shared_out_row0 + s * gs.shared_rows;
    }
    rows = rows < 0 ? 0 : rows;
    tb.rows[g] = rows;
    tb.a_row0[g] = arow;
    tb.out_row0[g] = orow;
    tb.tile_start[g + 1] = ((rows + BM - 1) / BM) * n_tiles;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int v = g < G ? tb.tile_start[g + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (g < G) tb.tile_start[g + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) tb.tile_start[0] = 0;
  }
  __syncthreads();
}

// MX FP8 activations keep every routed group's rows at a multiple of
// kPadRows (one CTA-pair tile): group g starts at kPadRows * (the blocks of
// kPadRows rows the groups before it need).
constexpr int kPadRows = 256;

// Sets a_row0 (bit 0 of `which`) and / or out_row0 (bit 1) of the routed
// groups to those padded starts.  Every thread of the block must call it.
__device__ __forceinline__ void pad_group_rows(GroupTable& tb, int E, int which) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int g = base + lane;
      const int blocks = g < E ? (tb.rows[g] + kPadRows - 1) / kPadRows : 0;
      int v = blocks;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (g < E) {
        const int start = (carry + v - blocks) * kPadRows;
        if (which & 1) tb.a_row0[g] = start;
        if (which & 2) tb.out_row0[g] = start;
      }
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
}

// Tile t (t < tile_start[G]) -> group g, row block and column block.
template <int BM>
__device__ __forceinline__ void decode_tile(const GroupTable& tb, int G, int t, int& g,
                                            int& m_blk, int& n_blk) {
  int lo = 0, hi = G;  // find g with tile_start[g] <= t < tile_start[g+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tb.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  g = lo;
  const int mt = (tb.rows[g] + BM - 1) / BM;
  const int local = t - tb.tile_start[g];
  n_blk = local / mt;
  m_blk = local - n_blk * mt;
}

}  // namespace moe
