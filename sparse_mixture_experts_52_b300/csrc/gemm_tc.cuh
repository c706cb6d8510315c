// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   out[row, n] = epilogue( sum_k A[a_row, k] * B_g[n, k] )   for every group g
//
// A is [rows, K] bf16 (K-major), B_g is expert g's nn.Linear weight [N, K]
// bf16 (K-major), accumulation is fp32 in tensor memory.  One persistent CTA
// per SM walks the tile list derived on the device from the dispatch offsets
// (groups.cuh).  Warp roles inside a CTA (192 threads):
//   warp 0     : TMA producer (one lane) - A and B tiles into a STAGES-deep ring
//   warp 1     : TMEM owner and MMA issuer (one lane) - 128 x BN x 16 MMAs
//   warps 2..5 : epilogue - tcgen05.ld, bias / activation, convert, store
//                (bf16 activations: the next GEMM's A operand; logits in fp32)
// The accumulator is double-buffered in TMEM (2 x BN fp32 columns) so the
// epilogue of one segment overlaps the main loop of the next.
//
// Work split.  Round-robin: CTA c takes whole tiles c, c + grid, ... so the
// CTAs running at the same time work on neighbouring tiles and share their
// weight slabs through L2.  With stream-K (the expert FFN) that holds for all
// whole waves but the last; the tiles left after them (one to two waves'
// worth, where whole tiles would leave SMs idle while the weights still
// stream) have their (tile, k-block) iterations flattened, and CTA c takes
// the contiguous range [c*W/P, (c+1)*W/P).  A CTA whose range starts inside a
// tile (only its first stream-K segment can) writes that segment's fp32
// partial to its slot and raises one flag per epilogue warp; the CTA that
// holds the tile's first k-block (the owner) adds the partials of the
// following CTAs in ascending order before its epilogue, so the result is the
// same on every run.  The following CTAs compute those pieces first, so the
// owner's waits are short.
//
// Overlapped projections.  The down-projection may start while the
// up-projection's last tiles still run: the up-projection's epilogue warps
// count, per expert group, the hidden tiles they have stored (ready[g], a
// release add after a proxy fence), and the down-projection's producer waits
// (acquire, bounded) until group g's count is complete before its first load
// of a g tile.  The down-projection then skips the grid-dependency wait at its
// start (it is launched once every up-projection CTA has passed its own, so
// the dispatch outputs it reads are complete) and waits for the up-projection
// grid at its end instead; its last CTA clears the counters.
//
// MX FP8 operands (MX = true).  A and B hold e4m3 codes; every 32 K-elements
// of every A row and B row share an E8M0 scale (the OCP Microscaling form).
// A stage then covers 128 K-elements (128 bytes per row, as a bf16 stage of
// 64), and brings, besides the two code boxes, one 512-byte block of scale
// bytes per 128 rows of A and of B (a bulk copy each).  Those blocks are
// stored pre-interleaved for the tensor core: byte (i, c, j) of a block, at
// offset 16 i + 4 c + j, is the scale of row 32 c + i for the stage's k-block
// j.  The MMA thread copies them into tensor memory (tcgen05.cp 32x128b,
// replicated into the four lane quarters), so that row m's scale for k-block
// j sits in lane m, column base + m / 32, byte j; the four k-blocks of a stage
// are four block-scaled MMAs of K = 32 selecting bytes 0..3.  The routed rows
// of A (and of a hidden activation the kernel writes) start at 256-row
// aligned ("padded") offsets (kPadRows), so every tile's rows are whole
// scale blocks.  An
// up-projection with MX output quantises its tile of the hidden activation in
// the epilogue: each thread holds one row, takes the largest magnitude of
// every 32 columns, and writes e4m3 codes plus the scale bytes.
//
// Every wait is bounded: a wait that runs out records MOE_DEV_ERR_* in the
// status word, raises the CTA abort flag, drains what this CTA has in flight
// and returns, so a bad launch can never hang the GPU.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "groups.cuh"
#include "ptx_sm100.cuh"

namespace moe {

// Epilogues: acc (+ bias) in fp32 (router logits, without bias; expert outputs
// kept in fp32); GELU(acc + b1) or SiLU(acc + b1) in bf16
// (up-projection); acc + b2 in bf16 (down-projection); the down-projection
// fused with the top-1 combine: out[token of the row] = w[token] * (acc + b2)
// in bf16; and SwiGLU, where the tile's BN accumulator columns are two halves
// - the gate projection's BN/2 columns, then the up projection's same BN/2
// columns (B rows n and N + n of a [2N, K] weight) - and the output is
// SiLU(gate) * up, BN/2 columns wide.
enum : int {
  EPI_F32 = 0,
  EPI_GELU_BF16 = 1,
  EPI_BIAS_BF16 = 2,
  EPI_SCATTER_BF16 = 3,
  EPI_SILU_BF16 = 4,
  EPI_SWIGLU_BF16 = 5,
  EPI_GELU_MX = 6,      // the activations of the up-projection, MX FP8 output
  EPI_SILU_MX = 7,
  EPI_SWIGLU_MX = 8
};
__host__ __device__ constexpr bool epi_glu(int e) { return e == EPI_SWIGLU_BF16 || e == EPI_SWIGLU_MX; }
__host__ __device__ constexpr bool epi_mx_out(int e) { return e >= EPI_GELU_MX; }
enum : int {
  DEV_ERR_WAIT_PRODUCER = 1,
  DEV_ERR_WAIT_MMA = 2,
  DEV_ERR_WAIT_EPILOGUE = 4,
  DEV_ERR_WAIT_PARTIAL = 16,
  DEV_ERR_WAIT_READY = 32
};
enum : int { READY_NONE = 0, READY_SIGNAL = 1, READY_WAIT = 2 };

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: any single wait
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s: draining after a give-up
constexpr int kMaxGemmCtas = 160;                  // stream-K partial slots (grid <= this)

struct TcArgs {
  GroupSpec gs;
  int N, K;
  void* out;                   // routed groups' rows
  void* out1;                  // shared groups' rows (row 0 of shared group 0)
  int64_t ldo;                 // elements between output rows
  const __nv_bfloat16* bias0;  // [E, N] or null
  const __nv_bfloat16* bias1;  // [n_shared, N] or null
  int* err;                    // device status word
  int streamk;                 // 1: stream-K split of the (tile, k-block) iterations
  float* partial;              // [kMaxGemmCtas][BN/16][128][16] fp32 (stream-K)
  int* flags;                  // [kMaxGemmCtas][4] zero between launches (stream-K)
  const int32_t* scatter_token;  // EPI_SCATTER_BF16: token of each output row
  const float* scatter_w;        // EPI_SCATTER_BF16: gate weight of each token (k = 1)
  int ready_mode;                // READY_*: overlapped up- and down-projections
  int* ready;                    // [groups] hidden-tile counters (zero between calls)
  unsigned int* ready_done;      // READY_WAIT: CTAs finished (zero between calls)
  int ready_up_tiles;            // READY_WAIT: column tiles of the up-projection per row tile
  // MX FP8 operands
  const uint8_t* sfa;            // A scale blocks [K/128][sfa_rb][512]
  int64_t sfa_rb;                // 128-row blocks of the (padded) A rows
  const uint8_t* sfb;            // B scale blocks [groups][K/128][sfb_nb][512]
  int sfb_nb;                    // 128-row blocks of one group's B rows
  uint8_t* sf_out;               // MX output: scale blocks [N/128][sf_out_rb][512]
  int64_t sf_out_rb;
  int pad_rows;                  // bit 0: routed A rows start at padded offsets; bit 1: output rows
};

__device__ __forceinline__ bool wait_timeout(uint64_t* bar, uint32_t parity, uint64_t limit) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ float gelu_erf(float v) {
  return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
}

// GELU for the epilogues that quantise their output to e4m3 (3 mantissa
// bits): erf by Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (Hastings' rational approximation, |error| <= 1.5e-7 for
// z >= 0): erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
// t = 1 / (1 + p z).  With e = 1 - erf(|v| / sqrt 2), GELU(v) = v (1 - e / 2)
// for v >= 0 and v e / 2 for v < 0 (no cancellation for negative v).  About a
// third of the instructions of erff; the error is far below an e4m3 step.
__device__ __forceinline__ float gelu_erf_as(float v) {
  const float z = fabsf(v) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f),
                       -0.284496736f),
               0.254829592f);
  const float e = poly * __expf(-z * z);
  return v >= 0.f ? v * fmaf(-0.5f, e, 1.0f) : 0.5f * v * e;
}

// v * sigmoid(v); for v -> -inf the quotient goes to -0, for v -> +inf to v
__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

// The segments (tile, [kb0, kb1)) a CTA processes, in order; every warp role
// walks the same sequence.
// Stream-K part of the split: tiles [dp_tiles, total) whose W = rem * KB
// iterations go to P = min(grid, W) CTAs, so every CTA below P has at least
// one iteration and the CTAs from P on have none.
struct SkSplit {
  int dp_tiles;   // tiles done round-robin before the stream-K part
  int64_t W;      // stream-K iterations
  int64_t P;      // CTAs sharing them
  __device__ void init(int total, int KB, int streamk) {
    const int G = gridDim.x;
    const int waves = total / G;
    // whole waves stay round-robin (concurrent CTAs share weight slabs in L2);
    // the last one to two waves' worth of tiles is split by iterations
    dp_tiles = !streamk ? total : (waves >= 2 ? (waves - 1) * G : 0);
    W = static_cast<int64_t>(total - dp_tiles) * KB;
    P = W < G ? W : G;
  }
  __device__ int64_t start(int64_t cta) const { return W * cta / P; }
};

struct SegIter {
  int t;             // next round-robin tile
  int64_t it, end;   // stream-K iterations of this CTA
  int dp_tiles, KB;
  __device__ void init(const SkSplit& sp, int kb) {
    KB = kb;
    dp_tiles = sp.dp_tiles;
    t = blockIdx.x;
    if (blockIdx.x < sp.P) {
      it = sp.start(blockIdx.x);
      end = sp.start(blockIdx.x + 1);
    } else {
      it = end = 0;
    }
  }
  __device__ bool next(int& tile, int& kb0, int& kb1) {
    if (t < dp_tiles) {
      tile = t;
      kb0 = 0;
      kb1 = KB;
      t += gridDim.x;
      return true;
    }
    if (it >= end) return false;
    const int64_t lt = it / KB;
    tile = dp_tiles + static_cast<int>(lt);
    kb0 = static_cast<int>(it - lt * KB);
    const int64_t rest = end - it;
    kb1 = (rest < KB - kb0) ? kb0 + static_cast<int>(rest) : KB;
    it += kb1 - kb0;
    return true;
  }
};

template <int BN, int STAGES, bool MX = false>
struct TcSmem {
  // a stage is 128 bytes of K per row: 64 bf16 or 128 e4m3 elements
  static constexpr int BM = 128, BK = MX ? 128 : 64;
  static constexpr uint32_t A_BYTES = BM * 128;
  static constexpr uint32_t B_BYTES = BN * 128;
  static constexpr uint32_t SF_BYTES = MX ? 512 * (1 + BN / 128) : 0;   // A, then B scale blocks
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
  // MX: the double-buffered accumulator, then a ring of scale columns (A at
  // 2 BN + 8 s, B at 2 BN + 64 + 8 s: 8-column aligned)
  static constexpr uint32_t TMEM_COLS = MX ? 512 : ((2 * BN < 32) ? 32 : 2 * BN);
  static constexpr uint32_t SFA_COL = 2 * BN, SFB_COL = 2 * BN + 64;
  static_assert(!MX || (BN == 128 && STAGES <= 8), "MX tiles: 128 wide, at most 8 stages");
  struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    GroupTable tb;
  };
  static constexpr size_t bytes() {
    return 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl);
  }
};

// The up-projection's epilogue with MX FP8 output, for one row of a tile
// (this thread's TMEM lane): the activation of the tile's BN accumulator
// columns (for SwiGLU the gate half times SiLU, the up half as the second
// factor), then per 32 output columns the largest magnitude, the E8M0 scale
// and the e4m3 codes, stored at row `orow` of the hidden activation, and the
// row's scale bytes in the interleaved block of its 128 rows and its
// 128-column stage.  The thread takes the tile's 32-column output blocks
// [cb0, cb1) (two warps share a lane quarter, each half the blocks).  `add`
// folds in stream-K partials of a 16-column chunk (a no-op without stream-K).
// Every lane of the warp must call it (the tensor-memory loads are
// warp-wide); `valid` only gates the stores.
template <int EPI, int BN, typename AddPartials>
__device__ __forceinline__ void mx_store_row(uint32_t trow, int n_blk, int cb0, int cb1, bool valid,
                                             int64_t orow, const __nv_bfloat16* bias,
                                             const TcArgs& args, AddPartials&& add) {
  constexpr bool GLU = epi_glu(EPI);
  constexpr int NCC = BN / 16;
  constexpr int BNO = GLU ? BN / 2 : BN;
  constexpr int NOUT = GLU ? NCC / 2 : NCC;
  static_assert(NOUT % 2 == 0, "whole 32-column blocks");
  uint32_t sfw = 0;   // the blocks' scale bytes, byte j = block j of the 128-column stage
#pragma unroll 1
  for (int cb = cb0; cb < cb1; ++cb) {
    float v[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int cc = 2 * cb + h;
      uint32_t r[16], ru[GLU ? 16 : 1];
      tmem_ld_32x32b_x16(trow + cc * 16, r);
      tmem_wait_ld(r);
      if constexpr (GLU) {
        tmem_ld_32x32b_x16(trow + (cc + NCC / 2) * 16, ru);
        tmem_wait_ld(ru);
      }
      const int col = n_blk * BNO + cc * 16;
      float a[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] = __uint_as_float(r[i]);
      add(cc, a);
      if (bias) {
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] += __bfloat162float(bias[col + i]);
      }
      if constexpr (GLU) {
        float u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = __uint_as_float(ru[i]);
        add(cc + NCC / 2, u);
        if (bias) {
#pragma unroll
          for (int i = 0; i < 16; ++i) u[i] += __bfloat162float(bias[args.N + col + i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = silu(a[i]) * u[i];
      } else if (EPI == EPI_SILU_MX) {
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = silu(a[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = gelu_erf_as(a[i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) v[16 * h + i] = a[i];
    }
    const int col = n_blk * BNO + cb * 32;
    if (!valid) continue;
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
    uint8_t* o = static_cast<uint8_t*>(args.out) + orow * args.ldo + col;
    *reinterpret_cast<uint4*>(o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4*>(o + 16) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    sfw |= sbyte << (8 * ((col >> 5) & 3));
  }
  if (valid) {   // this thread's blocks' bytes of the row's 4-byte scale word
    const int col0 = n_blk * BNO;
    uint8_t* sfp = args.sf_out +
                   ((static_cast<int64_t>(col0 >> 7) * args.sf_out_rb + (orow >> 7)) * 512) +
                   (orow & 31) * 16 + ((orow & 127) >> 5) * 4;
    for (int cb = cb0; cb < cb1; ++cb) {
      const int j = ((col0 + 32 * cb) >> 5) & 3;
      sfp[j] = static_cast<uint8_t>(sfw >> (8 * j));
    }
  }
}

// Epilogue warps: four, one per TMEM lane quarter; MX kernels take eight,
// two per lane quarter splitting the tile's columns (their quantising
// epilogue, alone on a scheduler, was the bottleneck of short-K tiles).
template <bool MX>
__host__ __device__ constexpr int tc_epi_warps() { return MX ? 8 : 4; }

template <int BN, int STAGES, int EPI, bool MX = false>
__global__ void __launch_bounds__(64 + 32 * tc_epi_warps<MX>(), 1)
k_gemm_tc(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
          const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
          const TcArgs args) {
  using L = TcSmem<BN, STAGES, MX>;
  constexpr int BM = L::BM, BK = L::BK;
  static_assert(!epi_mx_out(EPI) || MX, "an MX output comes from MX operands");
  constexpr int NCC = BN / 16;   // 16-column chunks of a tile
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert((BN & (BN - 1)) == 0, "TMEM columns must be a power of two");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  uint8_t* sSF = sB + STAGES * L::B_BYTES;   // MX scale blocks of every stage
  auto& c = *reinterpret_cast<typename L::Ctrl*>(smem + STAGES * L::STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GroupSpec& gs = args.gs;
  const int G = gs.E + gs.n_shared;
  constexpr bool GLU = epi_glu(EPI);
  constexpr bool MXO = epi_mx_out(EPI);
  constexpr int BNO = GLU ? BN / 2 : BN;   // output columns of a tile
  const int n_tiles = (args.N + BNO - 1) / BNO;
  const int KB = (args.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c.tfull[a], 1);
      mbar_init(&c.tempty[a], tc_epi_warps<MX>());
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
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, L::TMEM_COLS);
    tmem_relinquish();
  }
  // everything above overlaps the previous kernel's tail (programmatic launch);
  // an overlapped down-projection waits per group instead (see above)
  if (args.ready_mode != READY_WAIT) griddep_wait();
  griddep_launch_dependents();
  build_group_table<BM>(gs, n_tiles, c.tb);   // synchronises the block
  if (args.pad_rows) pad_group_rows(c.tb, gs.E, args.pad_rows);   // MX: padded group starts
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int total = c.tb.tile_start[G];
  volatile int* abort_flag = &c.abort_flag;
  SkSplit split;
  split.init(total, KB, MX ? 0 : args.streamk);   // MX: two warps a lane quarter, no stream-K
  SegIter seg;
  seg.init(split, KB);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) armed[s] = 0;
      bool ok = true;
      int ready_g = -1;   // last group whose hidden tiles are known complete
      int t, kb0, kb1;
      while (ok && seg.next(t, kb0, kb1)) {
        int g, m_blk, n_blk;
        decode_tile<BM>(c.tb, G, t, g, m_blk, n_blk);
        const bool routed = g < gs.E;
        const CUtensorMap* ma = (routed || gs.shared_a_sel == 0) ? &mA0 : &mA1;
        const CUtensorMap* mb = routed ? &mB0 : &mB1;
        const int bz = routed ? (gs.offsets ? g : 0) : g - gs.E;
        const int arow = c.tb.a_row0[g] + m_blk * BM;
        const int ncol = n_blk * BNO;
        if (args.ready_mode == READY_WAIT && g != ready_g) {
          // every hidden tile of group g stored by the up-projection (4 epilogue warps each)
          const int need =
              ((c.tb.rows[g] + BM - 1) / BM) * args.ready_up_tiles * tc_epi_warps<MX>();
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_gpu(args.ready + g) < need) {
            if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
              atomicOr(args.err, DEV_ERR_WAIT_READY);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          if (!ok) break;
          fence_proxy_async_global();   // the hidden rows are read by TMA (async proxy)
          ready_g = g;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(&c.empty[stage], phase ^ 1u, abort_flag, args.err,
                                 DEV_ERR_WAIT_PRODUCER, kWaitLimitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&c.full[stage], L::STAGE_BYTES);
          tma_load_2d(sA + stage * L::A_BYTES, ma, &c.full[stage], kb * BK, arow);
          if constexpr (MX) {
            // SwiGLU weights are packed with gate and up rows interleaved in
            // 64-row halves, so a tile's B rows are one box of BN rows
            const int brow = GLU ? n_blk * BN : ncol;
            tma_load_3d(sB + stage * L::B_BYTES, mb, &c.full[stage], kb * BK, brow, bz);
            uint8_t* sf = sSF + stage * L::SF_BYTES;
            bulk_load(sf, args.sfa + (static_cast<int64_t>(kb) * args.sfa_rb + arow / BM) * 512,
                      512, &c.full[stage]);
            bulk_load(sf + 512,
                      args.sfb + ((static_cast<int64_t>(bz) * KB + kb) * args.sfb_nb + brow / 128) * 512,
                      512, &c.full[stage]);
          } else {
            tma_load_3d(sB + stage * L::B_BYTES, mb, &c.full[stage], kb * BK, ncol, bz);
            if (GLU)   // the up projection's rows into the second half of the B tile
              tma_load_3d(sB + stage * L::B_BYTES + (BN / 2) * BK * 2, mb, &c.full[stage],
                          kb * BK, args.N + ncol, bz);
          }
#pragma unroll
          for (int s = 0; s < STAGES; ++s) armed[s] += (s == stage) ? 1u : 0u;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let every load already issued land before the CTA exits
#pragma unroll
        for (int s = 0; s < STAGES; ++s)
          if (armed[s]) wait_timeout(&c.full[s], (armed[s] - 1u) & 1u, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      int t, kb0, kb1;
      while (ok && seg.next(t, kb0, kb1)) {
        if (!mbar_wait_bounded(&c.tempty[acc], acc_phase ^ 1u, abort_flag, args.err,
                               DEV_ERR_WAIT_MMA, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(&c.full[stage], phase, abort_flag, args.err, DEV_ERR_WAIT_MMA,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * L::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * L::B_BYTES);
          if constexpr (MX) {
            // this stage's scale blocks into its tensor-memory columns, then
            // four block-scaled MMAs of K = 32 (bytes 0..3 of those columns)
            const uint32_t sf = smem_u32(sSF + stage * L::SF_BYTES);
            const uint32_t ta = tmem_base + L::SFA_COL + 8u * stage;
            const uint32_t tb = tmem_base + L::SFB_COL + 8u * stage;
            tmem_cp_32x128b_x4(ta, sdesc_sf_32x16(sf));
            tmem_cp_32x128b_x4(tb, sdesc_sf_32x16(sf + 512));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_mxf8(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32), sdesc_kmajor_sw128(b0 + kk * 32),
                        idesc_mxf8(BM, BN, kk, kk), ta, tb, (kb > kb0 || kk != 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              umma_bf16_f32(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32),
                            sdesc_kmajor_sw128(b0 + kk * 32), idesc,
                            (kb > kb0 || kk != 0) ? 1u : 0u);
            }
          }
          umma_commit(&c.empty[stage]);   // frees this smem stage once read
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&c.tfull[acc]);       // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok && issued) {  // wait for the MMAs in flight before TMEM is freed
        umma_commit(&c.drain);
        wait_timeout(&c.drain, 0, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = MX ? (warp - 2) >> 2 : 0;   // MX: which half of the tile's columns
    int acc = 0;
    uint32_t acc_phase = 0;
    int t, kb0, kb1;
    while (seg.next(t, kb0, kb1)) {
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
      const int row = q * 32 + lane;   // row of the tile this thread holds

      if (kb0 > 0) {
        // --------------------------------------------- a later piece of a tile:
        // fp32 partial to this CTA's slot, then this warp's flag
        float* slot = args.partial + static_cast<int64_t>(blockIdx.x) * NCC * BM * 16;
#pragma unroll 1
        for (int cc = 0; cc < NCC; ++cc) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(trow + cc * 16, r);
          tmem_wait_ld(r);
          float4* dst = reinterpret_cast<float4*>(slot + (static_cast<int64_t>(cc) * BM + row) * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&c.tempty[acc]);
          st_release_gpu(args.flags + blockIdx.x * 4 + q, 1);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }

      // --------------------------------------------- the tile's owner: if other
      // CTAs hold its later k-blocks (CTAs blockIdx+1 .. last), wait for their
      // partials (this warp's rows only)
      int last = blockIdx.x;
      if (kb1 < KB) {
        const int64_t tile_end = static_cast<int64_t>(t - split.dp_tiles + 1) * KB;
        while (last + 1 < split.P && split.start(last + 1) < tile_end) ++last;
        int good = 1;
        if (lane == 0) {
          for (int p = blockIdx.x + 1; p <= last && good; ++p) {
            const int* fl = args.flags + p * 4 + q;
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(fl) == 0) {
              if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
                atomicOr(args.err, DEV_ERR_WAIT_PARTIAL);
                *abort_flag = 1;
                good = 0;
                break;
              }
            }
            if (good) *const_cast<int*>(fl) = 0;   // consumed: zero for the next launch
          }
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        __syncwarp();
        if (!good) break;
      }

      const bool routed = g < gs.E;
      const int row_in_grp = m_blk * BM + row;
      const bool valid = row_in_grp < c.tb.rows[g];
      int64_t orow = static_cast<int64_t>(c.tb.out_row0[g]) + row_in_grp;
      float gate_w = 1.f;
      if (EPI == EPI_SCATTER_BF16 && valid) {   // the output row is the token's own row
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
      // later k-blocks of this tile from the following CTAs' partials, in order
      auto add_partials = [&](int chunk, float(&v)[16]) {
        for (int p = blockIdx.x + 1; p <= last; ++p) {
          const float4* src = reinterpret_cast<const float4*>(
              args.partial + (static_cast<int64_t>(p) * NCC * BM + static_cast<int64_t>(chunk) * BM + row) * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 w = __ldcg(src + i);
            v[4 * i] += w.x;
            v[4 * i + 1] += w.y;
            v[4 * i + 2] += w.z;
            v[4 * i + 3] += w.w;
          }
        }
      };
      constexpr int NOUT = GLU ? NCC / 2 : NCC;   // 16-column output chunks
      // 16-column output chunks of this warp: all, or (MX) its half
      const int cc_lo = MX ? half * (NOUT / 2) : 0;
      const int cc_hi = MX ? cc_lo + NOUT / 2 : NOUT;
      if constexpr (MXO)
        mx_store_row<EPI, BN>(trow, n_blk, cc_lo / 2, cc_hi / 2, valid, orow, bias, args,
                              add_partials);
#pragma unroll 1
      for (int cc = cc_lo; cc < (MXO ? cc_lo : cc_hi); ++cc) {
        uint32_t r[16], ru[GLU ? 16 : 1];
        tmem_ld_32x32b_x16(trow + cc * 16, r);
        tmem_wait_ld(r);
        if constexpr (GLU) {   // the up half's matching columns
          tmem_ld_32x32b_x16(trow + (cc + NCC / 2) * 16, ru);
          tmem_wait_ld(ru);
        }
        const int col = n_blk * BNO + cc * 16;
        if (!valid || col >= args.N) continue;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
        add_partials(cc, v);
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
        } else {
          if constexpr (GLU) {
            float w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __uint_as_float(ru[i]);
            add_partials(cc + NCC / 2, w);
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
      }
      if (args.ready_mode == READY_SIGNAL) {
        // this warp's rows of the tile are stored: count them for group g
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) red_add_release_gpu(args.ready + g, 1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
  if (args.ready_mode == READY_WAIT) {
    griddep_wait();   // this grid completes after the up-projection grid
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int prev;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "l"(args.ready_done)
                   : "memory");
      s_last = (prev == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {   // every CTA is past its waits: clear the counters for the next call
      for (int g = threadIdx.x; g < G; g += blockDim.x) args.ready[g] = 0;
      if (threadIdx.x == 0) *args.ready_done = 0u;
    }
  }
}

}  // namespace moe
