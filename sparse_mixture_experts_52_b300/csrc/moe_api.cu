// Host side of libmoe: argument validation, workspace layout, tensor-map
// construction and kernel launches behind the C ABI of include/moe.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "moe.h"
#include "dispatch.cuh"
#include "expert_choice.cuh"
#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "gemm_mx2.cuh"
#include "groups.cuh"
#include "mxfp8.cuh"
#include "route.cuh"
#include "route_tc.cuh"

using namespace moe;

namespace {

// ---------------------------------------------------------------- config
constexpr size_t kAlign = 256;
// workspace header (1 MiB at a fixed layout, zeroed by moe_workspace_init;
// every kernel leaves it zeroed again except the status word): the device
// status word at byte 0, the self-resetting block counters of the routing
// grid and of the standalone ranking grid, the per-expert assignment and
// arg-max totals, and the routing grid's per-block softmax partials
constexpr size_t kHeaderBytes = 1 << 20;
constexpr size_t kRouteCounterOffset = 16;
constexpr size_t kRankCounterOffset = 20;
constexpr size_t kStatsCounterOffset = 24;
constexpr size_t kReadyDoneOffset = 28;   // uint32: overlapped down-projection CTAs finished
constexpr size_t kTotalsOffset = 1024;    // int32 [E <= 256]
constexpr size_t kArgmaxOffset = 2048;    // uint32 [E <= 256]
constexpr size_t kFlagsOffset = 4096;     // int32 [kMaxGemmCtas][4] stream-K flags
constexpr size_t kReadyOffset = 8192;     // int32 [kMaxGroups] hidden tiles stored per group
constexpr size_t kPartOffset = 65536;     // fp32 [E + 1 <= 257, blocks <= 512]

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int next_pow2_min16(int v) {
  int p = 16;
  while (p < v) p <<= 1;
  return p;
}

inline size_t elem_bytes(const moe_config& c) { return c.dtype == MOE_BF16 ? 2 : 4; }
// expert outputs (y_perm, y_shared): the layer dtype, or fp32 when cfg.y_f32
inline size_t y_bytes(const moe_config& c) { return c.y_f32 ? 4 : elem_bytes(c); }

moe_status validate(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model <= 0 || c->d_ff <= 0) return MOE_ERR_INVALID_ARG;
  if (c->E < 1 || c->E > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > c->E || c->k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > kMaxShared) return MOE_ERR_INVALID_ARG;
  if (c->min_capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->route < MOE_ROUTE_SOFTMAX_TOPK || c->route > MOE_ROUTE_EXPERT_CHOICE)
    return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->aux_f != MOE_AUX_TOPK_COUNT && c->aux_f != MOE_AUX_ARGMAX) return MOE_ERR_INVALID_ARG;
  if (c->renorm != 0 && c->renorm != 1) return MOE_ERR_INVALID_ARG;
  if (c->has_bias != 0 && c->has_bias != 1) return MOE_ERR_INVALID_ARG;
  if (c->y_f32 != 0 && c->y_f32 != 1) return MOE_ERR_INVALID_ARG;
  if (c->expert_fmt != MOE_EXPERT_DENSE && c->expert_fmt != MOE_EXPERT_MXFP8)
    return MOE_ERR_INVALID_ARG;
  if (c->act < MOE_ACT_GELU || c->act > MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->capacity_factor) || !std::isfinite(c->aux_alpha))
    return MOE_ERR_INVALID_ARG;
  // Expert Choice needs a capacity: each expert takes C = floor(CF * T / E) tokens
  if (c->route == MOE_ROUTE_EXPERT_CHOICE && !(c->capacity_factor > 0.f))
    return MOE_ERR_INVALID_ARG;
  const int64_t Tk = static_cast<int64_t>(c->T) * c->k;
  const int64_t rows_ec = static_cast<int64_t>(c->E) * c->T;   // E * C <= E * T
  const int64_t rows_h = std::max(Tk, rows_ec) + static_cast<int64_t>(c->n_shared) * c->T;
  if (rows_h > (INT_MAX / 2)) return MOE_ERR_INVALID_ARG;
  // 16-byte rows for vector loads and TMA strides
  if (c->d_model % 8 != 0 || c->d_ff % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_F32 && c->E > 64) return MOE_ERR_UNSUPPORTED;
  if (c->expert_fmt == MOE_EXPERT_MXFP8 &&
      (c->dtype != MOE_BF16 || c->route == MOE_ROUTE_EXPERT_CHOICE || c->n_shared != 0 ||
       c->d_model % 128 != 0 || c->d_ff % 128 != 0))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool mx_experts(const moe_config& c) { return c.expert_fmt == MOE_EXPERT_MXFP8; }

// Rows of the MX activations: each expert's rows start at a multiple of kPadRows.
// 4 KB scale tile records of packed MX weights [G, N, K] (mxfp8.cuh)
int64_t mx_tile_records(int64_t G, int64_t N, int64_t K) { return G * (K / 128) * ((N + 255) / 256); }

int64_t mx_padded_rows(const moe_config& c) {
  return (static_cast<int64_t>(c.T) * c.k + (kPadRows - 1) * static_cast<int64_t>(c.E) +
          kPadRows - 1) / kPadRows * kPadRows;
}

int capacity_of(const moe_config& c) {
  if (!(c.capacity_factor > 0.f)) return INT_MAX;
  const double v = std::floor(static_cast<double>(c.capacity_factor) * c.T / c.E);
  int cap = v > static_cast<double>(INT_MAX / 2) ? INT_MAX / 2 : static_cast<int>(v);
  return std::max(cap, c.min_capacity);
}

bool expert_choice(const moe_config& c) { return c.route == MOE_ROUTE_EXPERT_CHOICE; }

// Tokens each expert takes under Expert Choice: the capacity, at most T.
int ec_capacity(const moe_config& c) { return std::min(capacity_of(c), c.T); }

// Expert-ordered rows the grouped FFN runs on: T*k assignments (top-k), or
// E*C (Expert Choice).
int64_t routed_rows(const moe_config& c) {
  return expert_choice(c) ? static_cast<int64_t>(c.E) * ec_capacity(c)
                          : static_cast<int64_t>(c.T) * c.k;
}

// bf16 routers over more than 64 experts or more tokens than the small-batch
// router takes run on the tensor cores
bool use_tc_router(const moe_config& c) {
  return c.dtype == MOE_BF16 && (c.E > 64 || c.T > kSmallRouteMaxT);
}

struct Layout {
  size_t status, logits, wgT, crank, hist;
  size_t idx, w, counts, kept, offsets, perm_token, slot_of, f, P, aux;
  size_t scoresT, tok_stats, ec_token, ec_w, ec_slot, ec_wt;   // Expert Choice
  size_t x_perm, H, Y, Ys, sk_part, total;
  size_t xq, xq_sf, hq, hq_sf;   // MX FP8 experts: codes and scale blocks (padded rows)
  int64_t mx_rows;
  int nb, E_pad;
  bool tc_router;   // the top-k router runs on the tensor cores
  bool tc_logits;   // the logits buffer and transposed W_g exist
};

Layout make_layout(const moe_config& c) {
  Layout L{};
  const size_t T = c.T, E = c.E, k = c.k, S = c.n_shared, d = c.d_model, F = c.d_ff;
  const size_t eb = elem_bytes(c);
  L.nb = route_blocks(c.T);
  L.E_pad = next_pow2_min16(c.E);
  L.tc_router = !expert_choice(c) && use_tc_router(c);
  L.tc_logits = c.dtype == MOE_BF16 && (L.tc_router || expert_choice(c));
  const bool ec = expert_choice(c);
  const size_t C = ec ? static_cast<size_t>(ec_capacity(c)) : 0;
  const size_t rows = static_cast<size_t>(routed_rows(c));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + std::max<size_t>(bytes, 1), kAlign);
    return at;
  };
  L.status = take(kHeaderBytes);
  static_assert(kPartOffset + size_t(kMaxExperts + 1) * (kRouteMaxBlocks > kSmallRouteMaxT
                                                         ? kRouteMaxBlocks
                                                         : kSmallRouteMaxT) * 4 <=
                    kHeaderBytes,
                "per-block partials must fit the header");
  L.logits = take(L.tc_logits ? T * L.E_pad * 4 : 0);
  L.wgT = take(L.tc_logits ? static_cast<size_t>(L.E_pad) * d * 2 : 0);
  L.crank = take(T * k * 4);
  L.hist = take(static_cast<size_t>(chunk_stride(c.T)) * E * 4);
  L.idx = take(T * k * 4);
  L.w = take(T * k * 4);
  L.counts = take(E * 4);
  L.kept = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm_token = take(T * k * 4);
  L.slot_of = take(T * k * 4);
  L.f = take(E * 4);
  L.P = take(E * 4);
  L.aux = take(4);
  L.scoresT = take(ec ? E * T * 4 : 0);
  L.tok_stats = take(ec ? 2 * T * 4 : 0);   // per-token softmax max, then sum
  L.ec_token = take(E * C * 4);
  L.ec_w = take(E * C * 4);
  L.ec_slot = take(ec ? E * T * 4 : 0);
  L.ec_wt = take(ec ? E * T * 4 : 0);
  L.x_perm = take(rows * d * eb);
  L.H = take((rows + S * T) * F * eb);
  L.Y = take(rows * d * y_bytes(c));
  L.Ys = take(S * T * d * y_bytes(c));
  // stream-K partial tiles of the tensor-core FFN: one 128 x 256 fp32 slot per CTA
  L.sk_part = take(c.dtype == MOE_BF16 ? static_cast<size_t>(kMaxGemmCtas) * 128 * 256 * 4 : 0);
  L.mx_rows = mx_experts(c) ? mx_padded_rows(c) : 0;
  const size_t mr = static_cast<size_t>(L.mx_rows);
  L.xq = take(mr * d);
  L.xq_sf = take(mr * d / 32);
  L.hq = take(mr * F);
  L.hq_sf = take(mr * F / 32);
  L.total = off;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

moe_status check_ws(const moe_config& c, void* ws, size_t ws_bytes, const Layout& L) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kAlign != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  (void)c;
  return MOE_OK;
}

// Launches `kern` with programmatic stream serialisation: it may begin while
// the previous kernel on the stream drains, and waits (griddep_wait) before
// it touches memory that kernel reads or writes.  Every kernel launched here
// starts with that wait.
template <typename... KArgs, typename... Args>
moe_status launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {0};
  if (dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [rows, K] bf16 row-major, box = 128 rows x 64 K, 128-byte swizzle
bool map_a(CUtensorMap* m, const void* base, int64_t K, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(std::max<int64_t>(rows, 1))};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [G, N, K] bf16, box = 1 x BN x 64, 128-byte swizzle
bool map_b(CUtensorMap* m, const void* base, int64_t K, int64_t N, int64_t G, int BN) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(std::max<int64_t>(G, 1))};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K * 2), static_cast<cuuint64_t>(N * K * 2)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MX FP8 codes [rows, K] bytes, box = 128 rows x 128 bytes, 128-byte swizzle
bool map_u8_a(CUtensorMap* m, const void* base, int64_t K, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(std::max<int64_t>(rows, 1))};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MX FP8 codes [G, N, K] bytes, box = 1 x box_rows x 128 bytes
bool map_u8_b(CUtensorMap* m, const void* base, int64_t K, int64_t N, int64_t G,
              int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(std::max<int64_t>(G, 1))};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N * K)};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MX scale blocks (n_blocks contiguous 512-byte blocks) as rows of 256 bytes;
// a box is `box_blocks` consecutive blocks (8: a 4 KB tile record), copied as
// they lie.  Wide rows keep a copy to few 256-byte requests.
bool map_sf_blocks(CUtensorMap* m, const void* base, int64_t n_blocks, int box_blocks = 1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(2 * std::max<int64_t>(n_blocks, 1))};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, static_cast<cuuint32_t>(2 * box_blocks)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- GEMM launch
template <int BN, int STAGES, int EPI, bool MX = false>
moe_status launch_tc_inst(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                          const CUtensorMap& b1, const TcArgs& args, int64_t row_tiles_ub,
                          cudaStream_t st) {
  constexpr size_t smem = TcSmem<BN, STAGES, MX>::bytes();
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(k_gemm_tc<BN, STAGES, EPI, MX>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  constexpr int BNO = epi_glu(EPI) ? BN / 2 : BN;   // output columns per tile
  const int64_t n_tiles = (args.N + BNO - 1) / BNO;
  const int64_t ub = std::max<int64_t>(1, row_tiles_ub * n_tiles);
  // stream-K: one CTA per SM (at most one partial slot each) whatever the tile
  // count; round-robin: no more CTAs than tiles
  const int grid = args.streamk ? std::min(num_sms(), kMaxGemmCtas)
                                : static_cast<int>(std::min<int64_t>(ub, num_sms()));
  return launch_pdl(k_gemm_tc<BN, STAGES, EPI, MX>, dim3(grid), dim3(64 + 32 * tc_epi_warps<MX>()),
                    smem, st, a0, a1, b0,
                    b1, args);
}

// The CTA-pair GEMM: clusters of two CTAs, as many clusters as can be
// resident at once (persistent; pairs of SMs, so an SM whose partner is busy
// or missing stays out), each pair taking 256-row tiles round robin.
template <int BN, int STAGES, int EPI>
moe_status launch_tc2_inst(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                           const CUtensorMap& b1, const TcArgs& args, int64_t pair_tiles_ub,
                           cudaStream_t st) {
  constexpr size_t smem = Tc2Smem<BN, STAGES>::bytes();
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
  if (max_pairs[dev] == 0) {
    if (cudaFuncSetAttribute(k_gemm_tc2<BN, STAGES, EPI>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    cfg.gridDim = dim3(2 * num_sms());
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc2<BN, STAGES, EPI>, &cfg) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    max_pairs[dev] = n;
  }
  const int64_t pairs = std::min<int64_t>(std::max<int64_t>(pair_tiles_ub, 1), max_pairs[dev]);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, k_gemm_tc2<BN, STAGES, EPI>, a0, a1, b0, b1, args) !=
      cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status launch_tc2(int epi, const CUtensorMap& a0, const CUtensorMap& a1,
                      const CUtensorMap& b0, const CUtensorMap& b1, const TcArgs& args,
                      int64_t pair_tiles_ub, cudaStream_t st) {
#define MOE_PAIR_EPI(EPI) \
  if (epi == EPI) return launch_tc2_inst<256, 6, EPI>(a0, a1, b0, b1, args, pair_tiles_ub, st);
  MOE_PAIR_EPI(EPI_GELU_BF16)
  MOE_PAIR_EPI(EPI_SILU_BF16)
  MOE_PAIR_EPI(EPI_SWIGLU_BF16)
  MOE_PAIR_EPI(EPI_BIAS_BF16)
  MOE_PAIR_EPI(EPI_F32)
  MOE_PAIR_EPI(EPI_SCATTER_BF16)
#undef MOE_PAIR_EPI
  return MOE_ERR_UNSUPPORTED;
}

// The block-scaled MX FP8 GEMMs on CTA pairs (gemm_mx2.cuh): 256 x 256 tiles,
// 6 stages of 33.5 KB a CTA, 320 threads; as many pairs as fit (persistent)
// up to the number of tiles.  sfa / sfb are the scale-block maps of A and B.
template <int STAGES, int EPI>
moe_status launch_mx2_inst(const CUtensorMap& a, const CUtensorMap& sfa, const CUtensorMap& b,
                           const CUtensorMap& sfb, const TcArgs& args, int64_t pair_tiles_ub,
                           cudaStream_t st) {
  constexpr size_t smem = Mx2Smem<STAGES>::bytes();
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
  if (max_pairs[dev] == 0) {
    if (cudaFuncSetAttribute(k_gemm_mx2<STAGES, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    cfg.gridDim = dim3(2 * num_sms());
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_mx2<STAGES, EPI>, &cfg) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    max_pairs[dev] = n;
  }
  const int64_t pairs = std::min<int64_t>(std::max<int64_t>(pair_tiles_ub, 1), max_pairs[dev]);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, k_gemm_mx2<STAGES, EPI>, a, sfa, b, sfb, args) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status launch_mx2(int epi, const CUtensorMap& a, const CUtensorMap& sfa, const CUtensorMap& b,
                      const CUtensorMap& sfb, const TcArgs& args, int64_t pair_tiles_ub,
                      cudaStream_t st) {
#define MOE_MX2_EPI(EPI) \
  if (epi == EPI) return launch_mx2_inst<6, EPI>(a, sfa, b, sfb, args, pair_tiles_ub, st);
  MOE_MX2_EPI(EPI_GELU_MX)
  MOE_MX2_EPI(EPI_SILU_MX)
  MOE_MX2_EPI(EPI_SWIGLU_MX)
  MOE_MX2_EPI(EPI_BIAS_BF16)
  MOE_MX2_EPI(EPI_F32)
  MOE_MX2_EPI(EPI_SCATTER_BF16)
#undef MOE_MX2_EPI
  return MOE_ERR_UNSUPPORTED;
}

// The block-scaled MX FP8 GEMMs: 128-wide tiles, 6 stages (33 KB each).
moe_status launch_tc_mx(int epi, const CUtensorMap& a0, const CUtensorMap& b0,
                        const TcArgs& args, int64_t row_tiles_ub, cudaStream_t st) {
#define MOE_MX_EPI(EPI) \
  if (epi == EPI) return launch_tc_inst<128, 6, EPI, true>(a0, a0, b0, b0, args, row_tiles_ub, st);
  MOE_MX_EPI(EPI_GELU_MX)
  MOE_MX_EPI(EPI_SILU_MX)
  MOE_MX_EPI(EPI_SWIGLU_MX)
  MOE_MX_EPI(EPI_BIAS_BF16)
  MOE_MX_EPI(EPI_F32)
  MOE_MX_EPI(EPI_SCATTER_BF16)
#undef MOE_MX_EPI
  return MOE_ERR_UNSUPPORTED;
}

// Row tiles (128 rows) of a grouped GEMM over n_rows expert-ordered rows in
// E groups, estimated on the host: the per-expert counts stay on the device.
int64_t est_row_tiles(int64_t n_rows, int E) {
  const int64_t dense = (n_rows + 127) / 128 + E / 2;    // plus ragged group tails
  return std::max<int64_t>(dense, std::min<int64_t>(E, n_rows));
}

// Tile width and work split of an expert-FFN GEMM.  With many waves of tiles
// (compute-bound layers) the split is stream-K over the last waves and the
// widest tile wins.  With few waves (weight streaming) whole tiles go round
// robin and the width is the one with the smallest estimated makespan: each
// round costs one tile, whose cost grows with BN (its weight slab) plus a
// fixed share for A and the epilogue (40 columns' worth, fitted on B300 with
// the projections overlapped: it takes 256-wide tiles for the Switch-shaped
// up-projection and 128-wide ones for the decode-shaped one, both faster in
// same-session A/B than the other choice).
struct FfnSplit {
  int bn, streamk;
};
FfnSplit pick_ffn_split(int N, int64_t row_tiles, int sms) {
  const int wide = N >= 256 ? 256 : (N >= 128 ? 128 : 64);
  const int64_t tiles_wide = row_tiles * ((N + wide - 1) / wide);
  if (tiles_wide >= 8 * static_cast<int64_t>(sms)) return FfnSplit{wide, 1};
  int best = wide;
  int64_t best_cost = INT64_MAX;
  for (int bn : {256, 128, 64}) {
    if (bn > wide) continue;
    const int64_t tiles = row_tiles * ((N + bn - 1) / bn);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const int64_t cost = rounds * (bn + 40);
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return FfnSplit{best, 0};
}

moe_status launch_tc(int epi, const CUtensorMap& a0, const CUtensorMap& a1,
                     const CUtensorMap& b0, const CUtensorMap& b1, const TcArgs& args, int BN,
                     int64_t row_tiles_ub, cudaStream_t st) {
  if (epi == EPI_F32) {
    switch (BN) {
      case 16: return launch_tc_inst<16, 8, EPI_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 32: return launch_tc_inst<32, 8, EPI_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 64: return launch_tc_inst<64, 8, EPI_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 128: return launch_tc_inst<128, 6, EPI_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 256: return launch_tc_inst<256, 4, EPI_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
    }
    return MOE_ERR_UNSUPPORTED;
  }
  // bf16 epilogues: tiles 64, 128 or 256 wide with 8, 6 or 4 pipeline stages
#define MOE_BF16_EPI(EPI)                                                                 \
  if (epi == EPI) {                                                                       \
    switch (BN) {                                                                         \
      case 64: return launch_tc_inst<64, 8, EPI>(a0, a1, b0, b1, args, row_tiles_ub, st);   \
      case 128: return launch_tc_inst<128, 6, EPI>(a0, a1, b0, b1, args, row_tiles_ub, st); \
      case 256: return launch_tc_inst<256, 4, EPI>(a0, a1, b0, b1, args, row_tiles_ub, st); \
    }                                                                                     \
    return MOE_ERR_UNSUPPORTED;                                                           \
  }
  MOE_BF16_EPI(EPI_GELU_BF16)
  MOE_BF16_EPI(EPI_BIAS_BF16)
  MOE_BF16_EPI(EPI_SCATTER_BF16)
  MOE_BF16_EPI(EPI_SILU_BF16)
  MOE_BF16_EPI(EPI_SWIGLU_BF16)
#undef MOE_BF16_EPI
  return MOE_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- steps
struct RouteOut {
  float* logits;
  int32_t* idx;
  float* w;
  float* f;
  float* P;
  float* aux;
  int32_t* counts;
  int32_t* kept;
  int32_t* offsets;
  float* z;
};

int kmax_of(int k) { return k <= 2 ? 2 : (k <= 4 ? 4 : (k <= 8 ? 8 : 16)); }

// The statistics reduction over nb per-block partials in the workspace header.
StatsArgs make_stats(const moe_config& c, void* ws, size_t status, int nb, const int32_t* counts,
                     float* f, float* P, float* aux, float* z) {
  StatsArgs sa{};
  sa.p_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + status + kPartOffset);
  sa.nb = nb;
  sa.a_tot = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + status + kArgmaxOffset);
  sa.counts = counts;
  sa.count_all = -1;
  sa.T = c.T;
  sa.E = c.E;
  sa.aux_f = c.aux_f;
  sa.alpha = c.aux_alpha;
  sa.f = f;
  sa.P = P;
  sa.aux = aux;
  sa.z = z;
  sa.done =
      reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + status + kStatsCounterOffset);
  return sa;
}

// Ranking state of a grid: chunk ranks and prefixes in `crank` / `hist`.
DispatchArgs dispatch_args(const moe_config& c, int32_t* crank, int32_t* hist, int32_t* totals,
                           int32_t* counts, int32_t* kept, int32_t* offsets, unsigned int* done,
                           int* err) {
  DispatchArgs dp{};
  dp.T = c.T;
  dp.k = c.k;
  dp.E = c.E;
  dp.C = capacity_of(c);
  dp.cpb = route_cpb(c.T);
  dp.crank = crank;
  dp.hist = hist;
  dp.totals = totals;
  dp.counts = counts;
  dp.kept = kept;
  dp.offsets = offsets;
  dp.done = done;
  dp.err = err;
  return dp;
}

template <int NPL>
moe_status launch_gate(int km, int nb, cudaStream_t st, const RouteArgs& ra) {
  constexpr int W = kGateWarps;
  switch (km) {
    case 2: return launch_pdl(k_gate<NPL, 2, W>, dim3(nb), dim3(W * 32), 0, st, ra);
    case 4: return launch_pdl(k_gate<NPL, 4, W>, dim3(nb), dim3(W * 32), 0, st, ra);
    case 8: return launch_pdl(k_gate<NPL, 8, W>, dim3(nb), dim3(W * 32), 0, st, ra);
    default: return launch_pdl(k_gate<NPL, 16, W>, dim3(nb), dim3(W * 32), 0, st, ra);
  }
}

template <typename TE, int EP>
moe_status launch_route_warp(int km, int nb, cudaStream_t st, const RouteArgs& ra, const TE* x,
                             const TE* w_g) {
  switch (km) {
    case 2: return launch_pdl(k_route_warp<TE, EP, 2>, dim3(nb), dim3(kRouteThreads), 0, st, ra, x, w_g);
    case 4: return launch_pdl(k_route_warp<TE, EP, 4>, dim3(nb), dim3(kRouteThreads), 0, st, ra, x, w_g);
    case 8: return launch_pdl(k_route_warp<TE, EP, 8>, dim3(nb), dim3(kRouteThreads), 0, st, ra, x, w_g);
    default: return launch_pdl(k_route_warp<TE, EP, 16>, dim3(nb), dim3(kRouteThreads), 0, st, ra, x, w_g);
  }
}

template <typename TE>
moe_status launch_route_warp_e(const moe_config& c, int nb, cudaStream_t st, const RouteArgs& ra,
                               const void* x, const void* w_g) {
  const int km = kmax_of(c.k);
  const auto* xt = static_cast<const TE*>(x);
  const auto* wt = static_cast<const TE*>(w_g);
  if (c.E <= 8) return launch_route_warp<TE, 8>(km, nb, st, ra, xt, wt);
  if (c.E <= 16) return launch_route_warp<TE, 16>(km, nb, st, ra, xt, wt);
  if (c.E <= 32) return launch_route_warp<TE, 32>(km, nb, st, ra, xt, wt);
  return launch_route_warp<TE, 64>(km, nb, st, ra, xt, wt);
}

template <typename TE, int EP>
moe_status launch_route_small(int km, int T, cudaStream_t st, const RouteArgs& ra, const TE* x,
                              const TE* w_g) {
  switch (km) {
    case 2: return launch_pdl(k_route_small<TE, EP, 2>, dim3(T), dim3(kRouteThreads), 0, st, ra, x, w_g);
    case 4: return launch_pdl(k_route_small<TE, EP, 4>, dim3(T), dim3(kRouteThreads), 0, st, ra, x, w_g);
    case 8: return launch_pdl(k_route_small<TE, EP, 8>, dim3(T), dim3(kRouteThreads), 0, st, ra, x, w_g);
    default: return launch_pdl(k_route_small<TE, EP, 16>, dim3(T), dim3(kRouteThreads), 0, st, ra, x, w_g);
  }
}

template <typename TE>
moe_status launch_route_small_e(const moe_config& c, cudaStream_t st, const RouteArgs& ra,
                                const void* x, const void* w_g) {
  const int km = kmax_of(c.k);
  const auto* xt = static_cast<const TE*>(x);
  const auto* wt = static_cast<const TE*>(w_g);
  if (c.E <= 8) return launch_route_small<TE, 8>(km, c.T, st, ra, xt, wt);
  if (c.E <= 16) return launch_route_small<TE, 16>(km, c.T, st, ra, xt, wt);
  if (c.E <= 32) return launch_route_small<TE, 32>(km, c.T, st, ra, xt, wt);
  return launch_route_small<TE, 64>(km, c.T, st, ra, xt, wt);
}

// The tensor-core router with the gating in its epilogue: bf16, E <= 16, and
// per-CTA softmax partials (one column per 128 tokens) that fit the header.
// Its epilogue gates one token per thread, serially over the experts; past 16
// experts that is slower on B300 than the separate gate kernel, which spreads
// a token's experts over a warp (measured: 36 vs 27 us of routing at T = 4096,
// E = 64).
int route_tc_split(const moe_config& c);

bool use_fused_tc_router(const moe_config& c) {
  const int64_t ctas = (static_cast<int64_t>(c.T) + 127) / 128;
  return use_tc_router(c) && c.E <= 16 &&
         ctas * (c.E + 1) <= static_cast<int64_t>(kMaxExperts + 1) * kRouteMaxRows &&
         route_tc_split(c) > 0;
}

// Blocks of the routing grid do_route launches (one per token for the
// small-batch router, one per 128 tokens for the fused tensor-core router).
int route_grid(const moe_config& c, const Layout& L) {
  if (!L.tc_router && c.T <= kSmallRouteMaxT) return c.T;
  if (use_fused_tc_router(c)) return (c.T + 127) / 128;
  return L.nb;
}

constexpr size_t kRouteTcMaxSmem = 232448 - 2048;   // opt-in shared memory less the static part
constexpr int kRouteTcMinStages = 4;

// Stages of the fused router's x ring: all the shared memory that the W_g
// slice, the partials and the control block leave, at most 12.
template <int S>
int route_tc_stages(int kbs) {
  using L = RouteTcSmem<S>;
  const size_t fixed = L::bytes(kbs, 0);
  if (fixed >= kRouteTcMaxSmem) return 0;
  return static_cast<int>(std::min<size_t>(L::kMaxStages, (kRouteTcMaxSmem - fixed) / L::A_BYTES));
}

// Cluster size of the fused router: enough CTAs per 128-token tile to cover
// the SMs, and enough for the tile's slice of W_g to leave room for at least
// four stages; 0 when no size in {1, 2, 4} does.
int route_tc_split(const moe_config& c) {
  const int tiles = (c.T + 127) / 128;
  const int KB = (c.d_model + 63) / 64;
  const int sms = num_sms();
  int s = tiles * 5 >= sms * 4 ? 1 : (tiles * 5 >= sms * 2 ? 2 : 4);
  while (s > 1 && s > KB) s /= 2;   // every rank gets a K block
  for (; s <= 4 && s <= std::max(KB, 1); s *= 2) {
    const int kbs = (KB + s - 1) / s;
    const int st = s == 1 ? route_tc_stages<1>(kbs)
                          : (s == 2 ? route_tc_stages<2>(kbs) : route_tc_stages<4>(kbs));
    if (st >= kRouteTcMinStages) return s;
  }
  return 0;
}

template <int KMAX, int S>
moe_status launch_route_tc_inst(const CUtensorMap& mx, const void* w_g, int w_vec, int tiles,
                                int KB, const RouteArgs& ra, cudaStream_t st) {
  const int kbs = (KB + S - 1) / S;
  const int stages = route_tc_stages<S>(kbs);
  if (stages < kRouteTcMinStages) return MOE_ERR_UNSUPPORTED;
  const size_t smem = RouteTcSmem<S>::bytes(kbs, stages);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(k_route_tc<KMAX, S>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kRouteTcMaxSmem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * S));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = S > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, k_route_tc<KMAX, S>, mx, static_cast<const __nv_bfloat16*>(w_g),
                         w_vec, stages, ra) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

template <int KMAX>
moe_status launch_route_tc_s(int split, const CUtensorMap& mx, const void* w_g, int w_vec,
                             int tiles, int KB, const RouteArgs& ra, cudaStream_t st) {
  if (split == 1) return launch_route_tc_inst<KMAX, 1>(mx, w_g, w_vec, tiles, KB, ra, st);
  if (split == 2) return launch_route_tc_inst<KMAX, 2>(mx, w_g, w_vec, tiles, KB, ra, st);
  return launch_route_tc_inst<KMAX, 4>(mx, w_g, w_vec, tiles, KB, ra, st);
}

moe_status launch_route_tc(int km, int split, const CUtensorMap& mx, const void* w_g, int w_vec,
                           int tiles, int KB, const RouteArgs& ra, cudaStream_t st) {
  switch (km) {
    case 2: return launch_route_tc_s<2>(split, mx, w_g, w_vec, tiles, KB, ra, st);
    case 4: return launch_route_tc_s<4>(split, mx, w_g, w_vec, tiles, KB, ra, st);
    case 8: return launch_route_tc_s<8>(split, mx, w_g, w_vec, tiles, KB, ra, st);
    default: return launch_route_tc_s<16>(split, mx, w_g, w_vec, tiles, KB, ra, st);
  }
}

// Router, gating, statistics and the dispatch ranking in one routing grid
// (plus the tensor-core router GEMM ahead of it for wide or long batches).
// logits [T, E_pad] fp32 in the workspace = x . W_g on the tensor cores, from
// the transposed W_g already in the workspace.  Expert columns go in tiles of
// at most 64: a wide router (E = 256) then spreads over four times as many
// CTAs as row tiles.
moe_status tc_logits_gemm(const moe_config& c, const Layout& L, void* ws, const void* x,
                          cudaStream_t st) {
  const int bn_r = std::min(L.E_pad, 64);
  CUtensorMap ma, mb;
  if (!map_a(&ma, x, c.d_model, c.T) ||
      !map_b(&mb, at<__nv_bfloat16>(ws, L.wgT), c.d_model, L.E_pad, 1, bn_r))
    return MOE_ERR_CUDA;
  float* logits_ws = at<float>(ws, L.logits);
  TcArgs ta{};
  ta.gs = GroupSpec{nullptr, 1, c.T, 0, 0, 0, 0, 0, 0};
  ta.N = L.E_pad;
  ta.K = c.d_model;
  ta.out = logits_ws;
  ta.out1 = logits_ws;
  ta.ldo = L.E_pad;
  ta.err = at<int>(ws, L.status);
  return launch_tc(EPI_F32, ma, ma, mb, mb, ta, bn_r, (c.T + 127) / 128 + 1, st);
}

moe_status do_route(const moe_config& c, const Layout& L, void* ws, const void* x,
                    const void* w_g, const float* lb, const float* sb, const RouteOut& o,
                    cudaStream_t st) {
  RouteArgs ra{};
  ra.T = c.T;
  ra.d = c.d_model;
  ra.E = c.E;
  ra.k = c.k;
  ra.route = c.route;
  ra.renorm = c.renorm;
  ra.logit_bias = lb;
  ra.select_bias = (c.route == MOE_ROUTE_BIASED_SOFTMAX) ? sb : nullptr;
  ra.logits_out = o.logits;
  ra.idx = o.idx;
  ra.w = o.w;
  ra.p_part = at<float>(ws, L.status + kPartOffset);
  ra.a_tot = at<unsigned int>(ws, L.status + kArgmaxOffset);
  ra.aux_f = c.aux_f;
  ra.alpha = c.aux_alpha;
  ra.f = o.f;
  ra.P = o.P;
  ra.aux = o.aux;
  ra.z = o.z;
  ra.dp = dispatch_args(c, at<int32_t>(ws, L.crank), at<int32_t>(ws, L.hist),
                        at<int32_t>(ws, L.status + kTotalsOffset), o.counts, o.kept, o.offsets,
                        at<unsigned int>(ws, L.status + kRouteCounterOffset),
                        at<int>(ws, L.status));
  const int nb = L.nb;
  const int km = kmax_of(c.k);
  moe_status s = MOE_OK;
  if (L.tc_router) {
    if (use_fused_tc_router(c)) {
      // a cluster of 1, 2 or 4 CTAs per 128 tokens (split over d), the gating
      // in the GEMM epilogue; W_g read as it is
      CUtensorMap mx;
      if (!map_a(&mx, x, c.d_model, c.T)) return MOE_ERR_CUDA;
      const int w_vec =
          (c.E == 8 || c.E == 16) && (reinterpret_cast<uintptr_t>(w_g) & 15) == 0 ? 1 : 0;
      return launch_route_tc(km, route_tc_split(c), mx, w_g, w_vec, (c.T + 127) / 128,
                             (c.d_model + 63) / 64, ra, st);
    }
    __nv_bfloat16* wgT = at<__nv_bfloat16>(ws, L.wgT);
    float* logits_ws = at<float>(ws, L.logits);
    dim3 tgrid((c.d_model + 31) / 32, (L.E_pad + 31) / 32);
    if ((s = launch_pdl(k_transpose_wg, tgrid, dim3(32, 8), 0, st,
                        static_cast<const __nv_bfloat16*>(w_g), c.d_model, c.E, L.E_pad, wgT)) !=
        MOE_OK)
      return s;
    if ((s = tc_logits_gemm(c, L, ws, x, st)) != MOE_OK) return s;
    ra.logits_in = logits_ws;
    ra.ld_in = L.E_pad;
    if (c.E <= 32) return launch_gate<1>(km, nb, st, ra);
    if (c.E <= 64) return launch_gate<2>(km, nb, st, ra);
    if (c.E <= 128) return launch_gate<4>(km, nb, st, ra);
    return launch_gate<8>(km, nb, st, ra);
  }
  if (c.T <= kSmallRouteMaxT) {
    if (c.dtype == MOE_BF16) return launch_route_small_e<__nv_bfloat16>(c, st, ra, x, w_g);
    return launch_route_small_e<float>(c, st, ra, x, w_g);
  }
  // fp32 batches beyond the small-batch router (bf16 ones take the tensor cores)
  return launch_route_warp_e<float>(c, nb, st, ra, x, w_g);
}

// ---------------------------------------------------------------- Expert Choice
struct EcOut {
  float* logits;      // [T, E] or null
  int32_t* ec_token;  // [E, C]
  float* ec_w;        // [E, C]
  int32_t* ec_slot;   // [E, T]
  float* ec_wt;       // [E, T] weight table for the combine, or null
  int32_t* offsets;   // [E + 1]
  int32_t* counts;    // [E] or null
  float *f, *P, *aux, *z;
};

int ec_scores_grid(const moe_config& c) {
  return std::max(1, std::min((c.T + kRouteWarps - 1) / kRouteWarps, kRouteMaxBlocks));
}

template <typename TE, int EP>
moe_status launch_ec_scores(int grid, const EcArgs& a, const void* x, const void* w_g,
                            cudaStream_t st) {
  constexpr int NPL = (EP + 31) / 32;
  return launch_pdl(k_ec_scores<TE, EP, NPL>, dim3(grid), dim3(kRouteThreads), 0, st, a,
                    static_cast<const TE*>(x), static_cast<const TE*>(w_g));
}

template <int NPL>
moe_status launch_ec_scores_from_logits(int grid, const EcArgs& a, cudaStream_t st) {
  return launch_pdl(k_ec_scores<__nv_bfloat16, 0, NPL>, dim3(grid), dim3(kRouteThreads), 0, st,
                    a, static_cast<const __nv_bfloat16*>(nullptr),
                    static_cast<const __nv_bfloat16*>(nullptr));
}

// Expert Choice routing: logits (tensor cores for bf16, CUDA cores for fp32),
// per-token softmax statistics, then one block per expert selects its tokens.
moe_status do_route_ec(const moe_config& c, const Layout& L, void* ws, const void* x,
                       const void* w_g, const float* lb, const EcOut& o, cudaStream_t st) {
  EcArgs a{};
  a.T = c.T;
  a.d = c.d_model;
  a.E = c.E;
  a.C = ec_capacity(c);
  a.logit_bias = lb;
  a.logits_out = o.logits;
  a.scoresT = at<float>(ws, L.scoresT);
  a.tok_max = at<float>(ws, L.tok_stats);
  a.tok_sum = at<float>(ws, L.tok_stats) + c.T;
  a.ec_token = o.ec_token;
  a.ec_w = o.ec_w;
  a.ec_slot = o.ec_slot;
  a.ec_wt = o.ec_wt;
  a.offsets = o.offsets;
  a.counts = o.counts;
  const int grid = ec_scores_grid(c);
  a.st = make_stats(c, ws, L.status, grid, nullptr, o.f, o.P, o.aux, o.z);
  a.st.count_all = a.C;   // every expert takes C tokens
  moe_status s;
  if (c.dtype == MOE_BF16) {
    dim3 tgrid((c.d_model + 31) / 32, (L.E_pad + 31) / 32);
    if ((s = launch_pdl(k_transpose_wg, tgrid, dim3(32, 8), 0, st,
                        static_cast<const __nv_bfloat16*>(w_g), c.d_model, c.E, L.E_pad,
                        at<__nv_bfloat16>(ws, L.wgT))) != MOE_OK)
      return s;
    if ((s = tc_logits_gemm(c, L, ws, x, st)) != MOE_OK) return s;
    a.logits_in = at<float>(ws, L.logits);
    a.ld_in = L.E_pad;
    if (c.E <= 32) s = launch_ec_scores_from_logits<1>(grid, a, st);
    else if (c.E <= 64) s = launch_ec_scores_from_logits<2>(grid, a, st);
    else if (c.E <= 128) s = launch_ec_scores_from_logits<4>(grid, a, st);
    else s = launch_ec_scores_from_logits<8>(grid, a, st);
  } else if (c.E <= 16) {
    s = launch_ec_scores<float, 16>(grid, a, x, w_g, st);
  } else if (c.E <= 32) {
    s = launch_ec_scores<float, 32>(grid, a, x, w_g, st);
  } else {
    s = launch_ec_scores<float, 64>(grid, a, x, w_g, st);
  }
  if (s != MOE_OK) return s;
  // one block per expert plus the statistics blocks; the column in registers
  // when it fits (up to 16 tokens a thread)
  const dim3 grid_sel(c.E + stats_blocks(c.E, kEcThreads / 32)), block_sel(kEcThreads);
  const int vpt = (c.T + kEcThreads - 1) / kEcThreads;
  if (vpt <= 4) return launch_pdl(k_ec_select_reg<4>, grid_sel, block_sel, 0, st, a);
  if (vpt <= 8) return launch_pdl(k_ec_select_reg<8>, grid_sel, block_sel, 0, st, a);
  if (vpt <= 16) return launch_pdl(k_ec_select_reg<16>, grid_sel, block_sel, 0, st, a);
  return launch_pdl(k_ec_select, grid_sel, block_sel, 0, st, a);
}

moe_status do_permute_ec(const moe_config& c, const void* x, const int32_t* ec_token,
                         int32_t* offsets, void* x_perm, cudaStream_t st) {
  const int C = ec_capacity(c);
  const int rows = c.E * C;
  const int grid = std::max(1, std::min((rows + 7) / 8, num_sms() * 8));
  return launch_pdl(k_ec_gather, dim3(grid), dim3(256), 0, st, ec_token, rows,
                    static_cast<int>(c.d_model * elem_bytes(c)), C, c.E,
                    static_cast<const uint8_t*>(x), static_cast<uint8_t*>(x_perm), offsets);
}

template <typename TY, typename TO, int U>
moe_status launch_ec_combine(const moe_config& c, int grid, const void* y_perm,
                             const int32_t* ec_slot, const float* ec_wt, const float* ec_w,
                             const void* y_shared, int S, void* out, cudaStream_t st) {
  auto go = [&](auto kern) {
    return launch_pdl(kern, dim3(grid), dim3(256), 0, st, static_cast<const TY*>(y_perm),
                      ec_slot, ec_wt, ec_w, static_cast<const TY*>(y_shared), S, c.T, c.E,
                      c.d_model, static_cast<TO*>(out));
  };
  if (c.E <= 64) return go(k_ec_combine<TY, TO, U, 2>);   // two groups of 32 experts per lane
  return go(k_ec_combine<TY, TO, U, kMaxExperts / 32>);
}

// bf16 rows: up to three 16-byte vectors per lane and pass (the whole row in
// one pass up to d = 768); fp32 rows: one (their loads take twice the registers)
moe_status launch_ec_combine_dt(const moe_config& c, int grid, const void* y_perm,
                                const int32_t* ec_slot, const float* ec_wt, const float* ec_w,
                                const void* y_shared, int S, void* out, cudaStream_t st) {
  if (c.dtype != MOE_BF16)
    return launch_ec_combine<float, float, 1>(c, grid, y_perm, ec_slot, ec_wt, ec_w, y_shared, S,
                                              out, st);
  using B = __nv_bfloat16;
  if (c.y_f32)   // fp32 expert outputs of a bf16 layer
    return launch_ec_combine<float, B, 1>(c, grid, y_perm, ec_slot, ec_wt, ec_w, y_shared, S,
                                          out, st);
  const int u = std::min(3, (c.d_model / 8 + 31) / 32);
  if (u <= 1) return launch_ec_combine<B, B, 1>(c, grid, y_perm, ec_slot, ec_wt, ec_w, y_shared, S, out, st);
  if (u == 2) return launch_ec_combine<B, B, 2>(c, grid, y_perm, ec_slot, ec_wt, ec_w, y_shared, S, out, st);
  return launch_ec_combine<B, B, 3>(c, grid, y_perm, ec_slot, ec_wt, ec_w, y_shared, S, out, st);
}

// ec_wt: the [E, T] weight table k_ec_select wrote in the workspace, or null
// (then the weights are read from the [E, C] list through the slots)
moe_status do_combine_ec(const moe_config& c, const void* y_perm, const int32_t* ec_slot,
                         const float* ec_w, const float* ec_wt, const void* y_shared, void* out,
                         cudaStream_t st) {
  const int grid = std::max(1, (c.T + 7) / 8);   // a warp per token
  const int S = y_shared ? c.n_shared : 0;
  return launch_ec_combine_dt(c, grid, y_perm, ec_slot, ec_wt, ec_w, y_shared, S, out, st);
}

// Slot resolution and row gather from the ranks a routing or ranking grid
// left.  Tokens per block: the largest of 32, 16, 8, 4 that still gives at
// least two blocks per SM.
// MX: x_perm receives MX FP8 codes at padded rows and xq_sf their scale
// blocks (sf_rb row blocks) instead of bf16 rows.
moe_status launch_permute(const moe_config& c, const int32_t* idx, const int32_t* crank,
                          const int32_t* hist, const int32_t* kept, const int32_t* offsets,
                          int32_t* perm_token, int32_t* slot_of, const void* x, void* x_perm,
                          cudaStream_t st, void* zero_out = nullptr,
                          const StatsArgs& stats = StatsArgs{}, uint8_t* xq_sf = nullptr,
                          int64_t sf_rb = 0) {
  const int row_bytes = c.d_model * static_cast<int>(elem_bytes(c));
  int tpb = 32;
  while (tpb > 4 && (c.T + tpb - 1) / tpb < 2 * num_sms()) tpb >>= 1;
  // plus the blocks of the routing statistics in a whole-layer pass
  const int grid =
      std::max(1, (c.T + tpb - 1) / tpb) + (stats.p_part ? stats_blocks(c.E, 8) : 0);
  const int ncs = chunk_stride(c.T);
  const auto* xb = static_cast<const uint8_t*>(x);
  auto* xp = static_cast<uint8_t*>(x_perm);
#define MOE_PERMUTE(KM, MXQ)                                                                \
  launch_pdl(k_permute<KM, MXQ>, dim3(grid), dim3(256), 0, st, idx, crank, hist, kept,      \
             offsets, c.T, c.k, c.E, ncs, tpb, row_bytes, xb, xp, perm_token, slot_of,     \
             static_cast<uint8_t*>(zero_out), stats, xq_sf, sf_rb)
  if (xq_sf) {
    switch (kmax_of(c.k)) {
      case 2: return MOE_PERMUTE(2, true);
      case 4: return MOE_PERMUTE(4, true);
      case 8: return MOE_PERMUTE(8, true);
      default: return MOE_PERMUTE(16, true);
    }
  }
  switch (kmax_of(c.k)) {
    case 2: return MOE_PERMUTE(2, false);
    case 4: return MOE_PERMUTE(4, false);
    case 8: return MOE_PERMUTE(8, false);
    default: return MOE_PERMUTE(16, false);
  }
#undef MOE_PERMUTE
}

// Ranking of caller-supplied indices, then the permute.
moe_status permute_from_idx(const moe_config& c, const DispatchArgs& dp, const void* x,
                            const int32_t* idx, int32_t* perm_token, int32_t* slot_of,
                            void* x_perm, cudaStream_t st) {
  const int nb = route_blocks(c.T);
  moe_status s;
  switch (kmax_of(c.k)) {
    case 2: s = launch_pdl(k_dispatch_rank<2>, dim3(nb), dim3(kRouteThreads), 0, st, dp, idx); break;
    case 4: s = launch_pdl(k_dispatch_rank<4>, dim3(nb), dim3(kRouteThreads), 0, st, dp, idx); break;
    case 8: s = launch_pdl(k_dispatch_rank<8>, dim3(nb), dim3(kRouteThreads), 0, st, dp, idx); break;
    default: s = launch_pdl(k_dispatch_rank<16>, dim3(nb), dim3(kRouteThreads), 0, st, dp, idx); break;
  }
  if (s != MOE_OK) return s;
  return launch_permute(c, idx, dp.crank, dp.hist, dp.kept, dp.offsets, perm_token, slot_of, x,
                        x_perm, st);
}

// ---------------------------------------------------------------- fixed scratch
// Scratch of moe_permute_noalloc: a file-scope device array, so that entry
// point needs no caller workspace and allocates nothing.  Host code must not
// pass `g_noalloc_scratch` itself to a kernel (in host code the name is only a
// host-side stand-in): the device address comes from cudaGetSymbolAddress,
// looked up on every call with the device current; the header is cleared
// whenever that address changes (the first call, or a new context after a
// device reset).  Layout in int32
// words: [0, 512) header (status word at 0, the ranking grid's block counter
// at 4 and the per-expert totals at [256, 512): all must start at zero), then
// the in-chunk ranks (T*k entries), then the per-chunk counts (E rows of
// ceil(T/32) rounded up to 32 entries).
constexpr int64_t kNoallocAssignments = MOE_PERMUTE_NOALLOC_MAX_ASSIGNMENTS;
constexpr int64_t kNoallocChunkCounts = MOE_PERMUTE_NOALLOC_MAX_CHUNK_COUNTS;
constexpr int64_t kNoallocHeader = 512;
constexpr int64_t kNoallocTotals = 256;
static __device__ __align__(256) int32_t
    g_noalloc_scratch[kNoallocHeader + kNoallocAssignments + kNoallocChunkCounts];

// Device address of g_noalloc_scratch on the current device, or null when the
// set-up fails.  Every call looks the address up (a host-side query); when it
// differs from the one this device had before -- the first call, or a new
// context after a device reset, whose copy of the array starts undefined --
// the header is cleared on `st`, stream ordered before the first use.
int32_t* noalloc_scratch(cudaStream_t st) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] != p) {
    if (cudaMemsetAsync(p, 0, kNoallocHeader * sizeof(int32_t), st) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return static_cast<int32_t*>(p);
}

struct FfnIn {
  const void *x_perm, *w1, *b1, *w2, *b2, *x, *ws1, *wsb1, *ws2, *wsb2;
  const int32_t* offsets;
  bool x_quantized;   // MX experts: the workspace already holds x_perm as MX FP8
};

// The top-1 combine fused into the down-projection (bf16, k = 1, no shared
// experts): each output row goes straight to out[token] scaled by the gate.
struct FfnScatter {
  void* out;                  // [T, d]
  const int32_t* perm_token;  // token of each expert-ordered row
  const float* w;             // [T] gate weights
};

// The grouped FFN on MX FP8 operands: the expert-ordered rows (quantised by
// the permute, or here from the caller's bf16 x_perm) and the hidden
// activation at kPadRows-aligned group offsets in the workspace, the packed
// weights, block-scaled tcgen05 MMAs.  Routed experts only.
moe_status do_ffn_mx(const moe_config& c, const Layout& L, void* ws, const FfnIn& in,
                     void* y_perm, cudaStream_t st, const FfnScatter* scatter) {
  const int64_t Tk = routed_rows(c);
  const int d = c.d_model, F = c.d_ff, E = c.E;
  const bool glu = c.act == MOE_ACT_SWIGLU;
  const int F1 = glu ? 2 * F : F;
  const int64_t R = L.mx_rows, RB = L.mx_rows / 128;
  uint8_t* xq = at<uint8_t>(ws, L.xq);
  uint8_t* xq_sf = at<uint8_t>(ws, L.xq_sf);
  uint8_t* hq = at<uint8_t>(ws, L.hq);
  uint8_t* hq_sf = at<uint8_t>(ws, L.hq_sf);
  moe_status s;
  if (!in.x_quantized) {
    const int grid = static_cast<int>(std::min<int64_t>((Tk + 7) / 8, num_sms() * 8));
    if ((s = launch_pdl(k_quant_rows_mx, dim3(std::max(grid, 1)), dim3(256), 0, st,
                        static_cast<const __nv_bfloat16*>(in.x_perm), in.offsets, E, d, RB, xq,
                        xq_sf)) != MOE_OK)
      return s;
  }
  const uint8_t* w1 = static_cast<const uint8_t*>(in.w1);
  const uint8_t* w2 = static_cast<const uint8_t*>(in.w2);
  // experts of 512 rows or more: CTA pairs with 256 x 256 tiles, when both
  // projections' weight rows are whole tiles
  const bool pair = Tk >= 512 * static_cast<int64_t>(E) && F1 % 256 == 0 && d % 256 == 0;
  const int b_rows = 128;
  CUtensorMap ma, mb, ha, hb, sxa, sw1, sha, sw2;
  if (!map_u8_a(&ma, xq, d, R) || !map_u8_b(&mb, w1, d, F1, E, b_rows) ||
      !map_u8_a(&ha, hq, F, R) || !map_u8_b(&hb, w2, F, d, E, b_rows))
    return MOE_ERR_CUDA;
  // the pair kernel loads the scale blocks with TMA: maps over them
  if (pair && (!map_sf_blocks(&sxa, xq_sf, (d / 128) * RB) ||
               !map_sf_blocks(&sw1, w1 + static_cast<int64_t>(E) * F1 * d * 33 / 32,
                              8 * mx_tile_records(E, F1, d), 8) ||
               !map_sf_blocks(&sha, hq_sf, (F / 128) * RB) ||
               !map_sf_blocks(&sw2, w2 + static_cast<int64_t>(E) * d * F * 33 / 32,
                              8 * mx_tile_records(E, d, F), 8)))
    return MOE_ERR_CUDA;
  const int64_t row_tiles_ub = (Tk + 127) / 128 + E;
  // whole tiles round robin (the MX kernels split no tile stream-K: their
  // eight epilogue warps share a lane quarter two by two)
  const bool sk_up = false, sk_dn = false;
  const bool overlap = !pair && !sk_up && !sk_dn;
  const int64_t pair_rows = (Tk + 255) / 256 + E;
  TcArgs up{};
  up.gs = GroupSpec{in.offsets, E, 0, 0, c.T, 0, 0, 0, 0};
  up.N = F;
  up.K = d;
  up.out = hq;
  up.out1 = hq;
  up.ldo = F;
  up.bias0 = static_cast<const __nv_bfloat16*>(c.has_bias ? in.b1 : nullptr);
  up.err = at<int>(ws, L.status);
  up.streamk = sk_up;
  up.partial = at<float>(ws, L.sk_part);
  up.flags = at<int>(ws, L.status + kFlagsOffset);
  up.sfa = xq_sf;
  up.sfa_rb = RB;
  up.sfb = w1 + static_cast<int64_t>(E) * F1 * d;
  up.sfb_nb = F1 / 128;
  up.sf_out = hq_sf;
  up.sf_out_rb = RB;
  up.pad_rows = 3;
  if (overlap) {
    up.ready_mode = READY_SIGNAL;
    up.ready = at<int>(ws, L.status + kReadyOffset);
  }
  const int epi_up = glu ? EPI_SWIGLU_MX : (c.act == MOE_ACT_SILU ? EPI_SILU_MX : EPI_GELU_MX);
  if ((s = pair ? launch_mx2(epi_up, ma, sxa, mb, sw1, up, pair_rows * (F1 / 256), st)
                : launch_tc_mx(epi_up, ma, mb, up, row_tiles_ub, st)) != MOE_OK)
    return s;
  TcArgs dn{};
  dn.gs = GroupSpec{in.offsets, E, 0, 0, c.T, 0, 0, 0, 0};
  dn.N = d;
  dn.K = F;
  dn.out = y_perm;
  dn.out1 = y_perm;
  dn.ldo = d;
  dn.bias0 = static_cast<const __nv_bfloat16*>(c.has_bias ? in.b2 : nullptr);
  dn.err = at<int>(ws, L.status);
  dn.streamk = sk_dn;
  dn.partial = at<float>(ws, L.sk_part);
  dn.flags = at<int>(ws, L.status + kFlagsOffset);
  dn.sfa = hq_sf;
  dn.sfa_rb = RB;
  dn.sfb = w2 + static_cast<int64_t>(E) * d * F;
  dn.sfb_nb = d / 128;
  dn.pad_rows = 1;
  if (overlap) {
    dn.ready_mode = READY_WAIT;
    dn.ready = at<int>(ws, L.status + kReadyOffset);
    dn.ready_done = at<unsigned int>(ws, L.status + kReadyDoneOffset);
    dn.ready_up_tiles = F / (glu ? 64 : 128);
  }
  const int epi_dn = scatter ? EPI_SCATTER_BF16 : (c.y_f32 ? EPI_F32 : EPI_BIAS_BF16);
  if (scatter) {
    dn.out = scatter->out;
    dn.scatter_token = scatter->perm_token;
    dn.scatter_w = scatter->w;
  }
  return pair ? launch_mx2(epi_dn, ha, sha, hb, sw2, dn, pair_rows * (d / 256), st)
              : launch_tc_mx(epi_dn, ha, hb, dn, row_tiles_ub, st);
}

// Experts holding 512 rows or more on average (compute-bound, many waves of
// tiles) run on CTA pairs with 256-row tiles; lighter ones on single CTAs,
// where a 256-row tile would be mostly empty.
bool use_pair_gemm(const moe_config& c) {
  return c.dtype == MOE_BF16 && !mx_experts(c) && routed_rows(c) >= 512 * static_cast<int64_t>(c.E);
}

// The grouped FFN on CTA pairs (bf16): whole 256 x 256 tiles round robin.
moe_status do_ffn_pair(const moe_config& c, const Layout& L, void* ws, const FfnIn& in,
                       void* y_perm, void* y_shared, cudaStream_t st, const FfnScatter* scatter) {
  const int64_t T = c.T, Tk = routed_rows(c), S = c.n_shared;
  const int d = c.d_model, F = c.d_ff;
  const bool glu = c.act == MOE_ACT_SWIGLU;
  const int F1 = glu ? 2 * F : F;
  void* H = at<uint8_t>(ws, L.H);
  void* H_shared = static_cast<uint8_t*>(H) + static_cast<size_t>(Tk) * F * 2;
  const int64_t pair_rows = (Tk + 255) / 256 + c.E + S * ((T + 255) / 256);
  CUtensorMap ma0, ma1, mb0, mb1;
  if (!map_a(&ma0, in.x_perm, d, std::max<int64_t>(Tk, 1)) || !map_b(&mb0, in.w1, d, F1, c.E, 128))
    return MOE_ERR_CUDA;
  if (S > 0) {
    if (!map_a(&ma1, in.x, d, T) || !map_b(&mb1, in.ws1, d, F1, S, 128)) return MOE_ERR_CUDA;
  } else {
    ma1 = ma0;
    mb1 = mb0;
  }
  TcArgs up{};
  up.gs = GroupSpec{in.offsets, c.E, 0, static_cast<int>(S), c.T, 1, 0, 0, 0};
  up.N = F;
  up.K = d;
  up.out = H;
  up.out1 = H_shared;
  up.ldo = F;
  up.bias0 = static_cast<const __nv_bfloat16*>(c.has_bias ? in.b1 : nullptr);
  up.bias1 = static_cast<const __nv_bfloat16*>(c.has_bias ? in.wsb1 : nullptr);
  up.err = at<int>(ws, L.status);
  const int epi_up = glu ? EPI_SWIGLU_BF16 : (c.act == MOE_ACT_SILU ? EPI_SILU_BF16 : EPI_GELU_BF16);
  moe_status s = launch_tc2(epi_up, ma0, ma1, mb0, mb1, up, pair_rows * ((F + (glu ? 127 : 255)) / (glu ? 128 : 256)), st);
  if (s != MOE_OK) return s;
  CUtensorMap ha, hb0, hb1;
  if (!map_a(&ha, H, F, Tk + S * T) || !map_b(&hb0, in.w2, F, d, c.E, 128)) return MOE_ERR_CUDA;
  if (S > 0) {
    if (!map_b(&hb1, in.ws2, F, d, S, 128)) return MOE_ERR_CUDA;
  } else {
    hb1 = hb0;
  }
  TcArgs dn{};
  dn.gs = GroupSpec{in.offsets, c.E, 0, static_cast<int>(S), c.T, 0, static_cast<int>(Tk), 0, c.T};
  dn.N = d;
  dn.K = F;
  dn.out = y_perm;
  dn.out1 = y_shared;
  dn.ldo = d;
  dn.bias0 = static_cast<const __nv_bfloat16*>(c.has_bias ? in.b2 : nullptr);
  dn.bias1 = static_cast<const __nv_bfloat16*>(c.has_bias ? in.wsb2 : nullptr);
  dn.err = at<int>(ws, L.status);
  const int64_t dn_tiles = pair_rows * ((d + 255) / 256);
  if (scatter) {
    dn.out = scatter->out;
    dn.scatter_token = scatter->perm_token;
    dn.scatter_w = scatter->w;
    return launch_tc2(EPI_SCATTER_BF16, ha, ha, hb0, hb1, dn, dn_tiles, st);
  }
  return launch_tc2(c.y_f32 ? EPI_F32 : EPI_BIAS_BF16, ha, ha, hb0, hb1, dn, dn_tiles, st);
}

moe_status do_ffn(const moe_config& c, const Layout& L, void* ws, const FfnIn& in, void* y_perm,
                  void* y_shared, cudaStream_t st, const FfnScatter* scatter = nullptr) {
  if (mx_experts(c)) return do_ffn_mx(c, L, ws, in, y_perm, st, scatter);
  if (use_pair_gemm(c)) return do_ffn_pair(c, L, ws, in, y_perm, y_shared, st, scatter);
  const int64_t T = c.T, Tk = routed_rows(c), S = c.n_shared;
  const int d = c.d_model, F = c.d_ff;
  void* H = at<uint8_t>(ws, L.H);
  const size_t eb = elem_bytes(c);
  void* H_shared = static_cast<uint8_t*>(H) + static_cast<size_t>(Tk) * F * eb;
  const int64_t row_tiles_ub = (Tk + S * T + 127) / 128 + c.E + S;
  const void* b1 = c.has_bias ? in.b1 : nullptr;
  const void* b2 = c.has_bias ? in.b2 : nullptr;
  const void* wsb1 = c.has_bias ? in.wsb1 : nullptr;
  const void* wsb2 = c.has_bias ? in.wsb2 : nullptr;
  moe_status s;
  const bool glu = c.act == MOE_ACT_SWIGLU;
  const int F1 = glu ? 2 * F : F;   // rows of W1: SwiGLU stacks the gate and up projections
  if (c.dtype == MOE_BF16) {
    CUtensorMap ma0, ma1, mb0, mb1;
    // up-projection + activation:  H = act(x_perm W1^T + b1)
    if (!map_a(&ma0, in.x_perm, d, std::max<int64_t>(Tk, 1))) return MOE_ERR_CUDA;
    const int64_t rt = est_row_tiles(Tk, c.E) + S * ((T + 127) / 128);
    const FfnSplit sp_up = pick_ffn_split(F1, rt, num_sms());
    const int bn_up = sp_up.bn;
    // SwiGLU: each B tile is two boxes of bn_up / 2 rows (gate rows n.., up rows F + n..)
    const int box_up = glu ? bn_up / 2 : bn_up;
    if (!map_b(&mb0, in.w1, d, F1, c.E, box_up)) return MOE_ERR_CUDA;
    if (S > 0) {
      if (!map_a(&ma1, in.x, d, T) || !map_b(&mb1, in.ws1, d, F1, S, box_up)) return MOE_ERR_CUDA;
    } else {
      ma1 = ma0;
      mb1 = mb0;
    }
    static_assert(kFlagsOffset + kMaxGemmCtas * 4 * sizeof(int) <= kReadyOffset, "header layout");
    static_assert(kReadyOffset + kMaxGroups * sizeof(int) <= kPartOffset, "header layout");
    TcArgs up{};
    up.gs = GroupSpec{in.offsets, c.E, 0, static_cast<int>(S), c.T, 1, 0, 0, 0};
    up.N = F;
    up.K = d;
    up.out = H;
    up.out1 = H_shared;
    up.ldo = F;
    up.bias0 = static_cast<const __nv_bfloat16*>(b1);
    up.bias1 = static_cast<const __nv_bfloat16*>(wsb1);
    up.err = at<int>(ws, L.status);
    up.streamk = sp_up.streamk;
    up.partial = at<float>(ws, L.sk_part);
    up.flags = at<int>(ws, L.status + kFlagsOffset);
    // the down-projection may overlap the up-projection's last tiles when
    // neither splits tiles stream-K (they would share the partial slots)
    const FfnSplit sp_dn = pick_ffn_split(d, rt, num_sms());
    const bool overlap = !sp_up.streamk && !sp_dn.streamk;
    if (overlap) {
      up.ready_mode = READY_SIGNAL;
      up.ready = at<int>(ws, L.status + kReadyOffset);
    }
    const int epi_up = glu ? EPI_SWIGLU_BF16
                           : (c.act == MOE_ACT_SILU ? EPI_SILU_BF16 : EPI_GELU_BF16);
    if ((s = launch_tc(epi_up, ma0, ma1, mb0, mb1, up, bn_up, row_tiles_ub, st)) != MOE_OK)
      return s;
    // down-projection:  y = H W2^T + b2
    CUtensorMap ha, hb0, hb1;
    if (!map_a(&ha, H, F, Tk + S * T)) return MOE_ERR_CUDA;
    const int bn_dn = sp_dn.bn;
    if (!map_b(&hb0, in.w2, F, d, c.E, bn_dn)) return MOE_ERR_CUDA;
    if (S > 0) {
      if (!map_b(&hb1, in.ws2, F, d, S, bn_dn)) return MOE_ERR_CUDA;
    } else {
      hb1 = hb0;
    }
    TcArgs dn{};
    dn.gs = GroupSpec{in.offsets, c.E, 0, static_cast<int>(S), c.T, 0, static_cast<int>(Tk), 0, c.T};
    dn.N = d;
    dn.K = F;
    dn.out = y_perm;
    dn.out1 = y_shared;
    dn.ldo = d;
    dn.bias0 = static_cast<const __nv_bfloat16*>(b2);
    dn.bias1 = static_cast<const __nv_bfloat16*>(wsb2);
    dn.err = at<int>(ws, L.status);
    dn.streamk = sp_dn.streamk;
    dn.partial = at<float>(ws, L.sk_part);
    dn.flags = at<int>(ws, L.status + kFlagsOffset);
    if (overlap) {
      dn.ready_mode = READY_WAIT;
      dn.ready = at<int>(ws, L.status + kReadyOffset);
      dn.ready_done = at<unsigned int>(ws, L.status + kReadyDoneOffset);
      const int bno_up = glu ? bn_up / 2 : bn_up;   // output columns of an up-projection tile
      dn.ready_up_tiles = (F + bno_up - 1) / bno_up;
    }
    if (scatter) {
      dn.out = scatter->out;
      dn.scatter_token = scatter->perm_token;
      dn.scatter_w = scatter->w;
      return launch_tc(EPI_SCATTER_BF16, ha, ha, hb0, hb1, dn, bn_dn, row_tiles_ub, st);
    }
    return launch_tc(c.y_f32 ? EPI_F32 : EPI_BIAS_BF16, ha, ha, hb0, hb1, dn, bn_dn,
                     row_tiles_ub, st);
  }
  // fp32: CUDA-core grouped GEMMs
  const int64_t tiles_ub = (Tk + S * T + 63) / 64 + c.E + S;
  SimtArgs up{};
  up.gs = GroupSpec{in.offsets, c.E, 0, static_cast<int>(S), c.T, 1, 0, 0, 0};
  up.N = F;
  up.K = d;
  up.A0 = static_cast<const float*>(in.x_perm);
  up.A1 = static_cast<const float*>(in.x);
  up.lda = d;
  up.B0 = static_cast<const float*>(in.w1);
  up.B1 = static_cast<const float*>(in.ws1);
  up.bias0 = static_cast<const float*>(b1);
  up.bias1 = static_cast<const float*>(wsb1);
  up.out = static_cast<float*>(H);
  up.out1 = static_cast<float*>(H_shared);
  up.ldo = F;
  up.act = glu ? SIMT_ACT_SWIGLU : (c.act == MOE_ACT_SILU ? SIMT_ACT_SILU : SIMT_ACT_GELU);
  int grid = static_cast<int>(std::min<int64_t>(tiles_ub * ((F + 63) / 64), num_sms() * 4));
  s = glu ? launch_pdl(k_gemm_simt_f32<true>, dim3(std::max(grid, 1)), dim3(256), 0, st, up)
          : launch_pdl(k_gemm_simt_f32<false>, dim3(std::max(grid, 1)), dim3(256), 0, st, up);
  if (s != MOE_OK) return s;
  SimtArgs dn{};
  dn.gs = GroupSpec{in.offsets, c.E, 0, static_cast<int>(S), c.T, 0, static_cast<int>(Tk), 0, c.T};
  dn.N = d;
  dn.K = F;
  dn.A0 = static_cast<const float*>(H);
  dn.A1 = static_cast<const float*>(H);
  dn.lda = F;
  dn.B0 = static_cast<const float*>(in.w2);
  dn.B1 = static_cast<const float*>(in.ws2);
  dn.bias0 = static_cast<const float*>(b2);
  dn.bias1 = static_cast<const float*>(wsb2);
  dn.out = static_cast<float*>(y_perm);
  dn.out1 = static_cast<float*>(y_shared);
  dn.ldo = d;
  dn.act = SIMT_ACT_NONE;
  grid = static_cast<int>(std::min<int64_t>(tiles_ub * ((d + 63) / 64), num_sms() * 4));
  return launch_pdl(k_gemm_simt_f32<false>, dim3(std::max(grid, 1)), dim3(256), 0, st, dn);
}

moe_status do_combine(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                      const float* w, const void* y_shared, void* out, cudaStream_t st) {
  const int grid = std::max(1, std::min((c.T + 7) / 8, num_sms() * 8));
  const int S = y_shared ? c.n_shared : 0;
  // U 16-byte vectors per lane and pass: two for bf16 top-1/2 and top-3/4 rows,
  // one with more slots in flight (or fp32 rows)
#define MOE_COMBINE(TY, TO, KM, U)                                                          \
  return launch_pdl(k_combine<TY, TO, KM, U>, dim3(grid), dim3(256), 0, st,                 \
                    static_cast<const TY*>(y_perm), slot_of, w,                             \
                    static_cast<const TY*>(y_shared), S, c.T, c.k, c.d_model,                \
                    static_cast<TO*>(out))
  const int km = kmax_of(c.k);
  using B = __nv_bfloat16;
  if (c.dtype == MOE_BF16 && !c.y_f32) {
    if (km == 2) MOE_COMBINE(B, B, 2, 2);
    if (km == 4) MOE_COMBINE(B, B, 4, 2);
    if (km == 8) MOE_COMBINE(B, B, 8, 1);
    MOE_COMBINE(B, B, 16, 1);
  }
  if (c.dtype == MOE_BF16) {   // fp32 expert outputs, bf16 layer output
    if (km == 2) MOE_COMBINE(float, B, 2, 1);
    if (km == 4) MOE_COMBINE(float, B, 4, 1);
    if (km == 8) MOE_COMBINE(float, B, 8, 1);
    MOE_COMBINE(float, B, 16, 1);
  }
  if (km == 2) MOE_COMBINE(float, float, 2, 1);
  if (km == 4) MOE_COMBINE(float, float, 4, 1);
  if (km == 8) MOE_COMBINE(float, float, 8, 1);
  MOE_COMBINE(float, float, 16, 1);
#undef MOE_COMBINE
}

moe_status zero_stats(const moe_config& c, int32_t* counts, float* f, float* P, float* aux,
                      int32_t* offsets, int32_t* kept, cudaStream_t st) {
  const size_t E = c.E;
  if (counts && cudaMemsetAsync(counts, 0, E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (kept && cudaMemsetAsync(kept, 0, E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (offsets && cudaMemsetAsync(offsets, 0, (E + 1) * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (f && cudaMemsetAsync(f, 0, E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (P && cudaMemsetAsync(P, 0, E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (aux && cudaMemsetAsync(aux, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream stream) {
  if (!ws || ws_bytes < kHeaderBytes || reinterpret_cast<uintptr_t>(ws) % kAlign != 0)
    return MOE_ERR_WORKSPACE;
  return cudaMemsetAsync(ws, 0, kHeaderBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* w_g,
                     const float* logit_bias, const float* select_bias, float* logits,
                     int32_t* topk_idx, float* topk_w, float* f, float* P, float* aux,
                     float* z_loss, void* ws, size_t ws_bytes, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if ((s = check_ws(c, ws, ws_bytes, L)) != MOE_OK) return s;
  if (expert_choice(c)) return MOE_ERR_INVALID_ARG;   // moe_route_expert_choice
  if (!f || !P || !aux) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    if (z_loss && cudaMemsetAsync(z_loss, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    return zero_stats(c, nullptr, f, P, aux, nullptr, nullptr, st);
  }
  if (!x || !w_g || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((s = do_route(c, L, ws, x, w_g, logit_bias, select_bias,
                    RouteOut{logits, topk_idx, topk_w, f, P, aux, at<int32_t>(ws, L.counts),
                             at<int32_t>(ws, L.kept), at<int32_t>(ws, L.offsets), z_loss},
                    st)) != MOE_OK)
    return s;
  // the routing statistics: a small grid of their own after the routing grid
  const StatsArgs sa =
      make_stats(c, ws, L.status, route_grid(c, L), at<int32_t>(ws, L.counts), f, P, aux, z_loss);
  return launch_pdl(k_stats, dim3(stats_blocks(c.E, 8)), dim3(256), 0, st, sa);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* perm_token,
                       int32_t* slot_of, void* x_perm, void* ws, size_t ws_bytes,
                       moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if ((s = check_ws(c, ws, ws_bytes, L)) != MOE_OK) return s;
  if (expert_choice(c)) return MOE_ERR_INVALID_ARG;   // moe_permute_expert_choice
  if (!counts || !kept || !offsets) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return zero_stats(c, counts, nullptr, nullptr, nullptr, offsets, kept, st);
  if (!x || !topk_idx || !perm_token || !slot_of || !x_perm) return MOE_ERR_INVALID_ARG;
  const DispatchArgs dp = dispatch_args(c, at<int32_t>(ws, L.crank), at<int32_t>(ws, L.hist),
                                        at<int32_t>(ws, L.status + kTotalsOffset), counts, kept,
                                        offsets,
                                        at<unsigned int>(ws, L.status + kRankCounterOffset),
                                        at<int>(ws, L.status));
  return permute_from_idx(c, dp, x, topk_idx, perm_token, slot_of, x_perm, st);
}

moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               int32_t* counts, int32_t* kept, int32_t* offsets,
                               int32_t* perm_token, int32_t* slot_of, void* x_perm,
                               moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(c.T) * c.k > kNoallocAssignments ||
      static_cast<int64_t>(chunk_stride(c.T)) * c.E > kNoallocChunkCounts)
    return MOE_ERR_UNSUPPORTED;
  if (!counts || !kept || !offsets) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return zero_stats(c, counts, nullptr, nullptr, nullptr, offsets, kept, st);
  if (!x || !topk_idx || !perm_token || !slot_of || !x_perm) return MOE_ERR_INVALID_ARG;
  int32_t* scratch = noalloc_scratch(st);
  if (!scratch) return MOE_ERR_CUDA;
  const DispatchArgs dp =
      dispatch_args(c, scratch + kNoallocHeader, scratch + kNoallocHeader + kNoallocAssignments,
                    scratch + kNoallocTotals, counts, kept, offsets,
                    reinterpret_cast<unsigned int*>(scratch + 4), scratch);
  return permute_from_idx(c, dp, x, topk_idx, perm_token, slot_of, x_perm, st);
}

moe_status moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                           const void* w1, const void* b1, const void* w2, const void* b2,
                           const void* x, const void* ws1, const void* wsb1, const void* ws2,
                           const void* wsb2, void* y_perm, void* y_shared, void* ws,
                           size_t ws_bytes, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if ((s = check_ws(c, ws, ws_bytes, L)) != MOE_OK) return s;
  if (c.T == 0) return MOE_OK;
  if (!x_perm || !offsets || !w1 || !w2 || !y_perm) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (!x || !ws1 || !ws2 || !y_shared)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && c.has_bias && (!wsb1 || !wsb2)) return MOE_ERR_INVALID_ARG;
  FfnIn in{x_perm, w1, b1, w2, b2, x, ws1, wsb1, ws2, wsb2, offsets};
  return do_ffn(c, L, ws, in, y_perm, y_shared, static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot_of,
                       const float* topk_w, const void* y_shared, void* out, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_INVALID_ARG;   // moe_combine_expert_choice
  if (c.T == 0) return MOE_OK;
  if (!y_perm || !slot_of || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
  return do_combine(c, y_perm, slot_of, topk_w, c.n_shared > 0 ? y_shared : nullptr, out,
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_forward(const moe_config* cfg, const void* x, const void* w_g,
                       const float* logit_bias, const float* select_bias, const void* w1,
                       const void* b1, const void* w2, const void* b2, const void* ws1,
                       const void* wsb1, const void* ws2, const void* wsb2, void* out,
                       int32_t* topk_idx, float* topk_w, int32_t* counts, float* f, float* P,
                       float* aux, float* z_loss, void* ws, size_t ws_bytes, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if ((s = check_ws(c, ws, ws_bytes, L)) != MOE_OK) return s;
  if (!out && c.T > 0) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.idx);
  float* w = topk_w ? topk_w : at<float>(ws, L.w);
  int32_t* cnt = counts ? counts : at<int32_t>(ws, L.counts);
  float* fo = f ? f : at<float>(ws, L.f);
  float* Po = P ? P : at<float>(ws, L.P);
  float* ao = aux ? aux : at<float>(ws, L.aux);
  if (c.T == 0) {
    if (z_loss && cudaMemsetAsync(z_loss, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    return zero_stats(c, counts, f, P, aux, nullptr, nullptr, st);
  }
  if (!x || !w_g || !w1 || !w2) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (!ws1 || !ws2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && c.has_bias && (!wsb1 || !wsb2)) return MOE_ERR_INVALID_ARG;
  void* Y = at<uint8_t>(ws, L.Y);
  void* Ys = at<uint8_t>(ws, L.Ys);

  if (expert_choice(c)) {
    // topk_idx / topk_w carry the [E, C] taken tokens and their weights
    int32_t* tok = topk_idx ? topk_idx : at<int32_t>(ws, L.ec_token);
    float* ew = topk_w ? topk_w : at<float>(ws, L.ec_w);
    int32_t* slot = at<int32_t>(ws, L.ec_slot);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    void* x_perm = at<uint8_t>(ws, L.x_perm);
    if ((s = do_route_ec(c, L, ws, x, w_g, logit_bias,
                         EcOut{nullptr, tok, ew, slot, at<float>(ws, L.ec_wt), offsets, cnt, fo,
                               Po, ao, z_loss},
                         st)) !=
        MOE_OK)
      return s;
    if ((s = do_permute_ec(c, x, tok, offsets, x_perm, st)) != MOE_OK) return s;
    FfnIn in{x_perm, w1, b1, w2, b2, x, ws1, wsb1, ws2, wsb2, offsets};
    if ((s = do_ffn(c, L, ws, in, Y, Ys, st)) != MOE_OK) return s;
    return do_combine_ec(c, Y, slot, ew, at<float>(ws, L.ec_wt),
                         c.n_shared > 0 ? Ys : nullptr, out, st);
  }

  int32_t* kept = at<int32_t>(ws, L.kept);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* slot_of = at<int32_t>(ws, L.slot_of);
  int32_t* perm_token = at<int32_t>(ws, L.perm_token);
  void* x_perm = at<uint8_t>(ws, L.x_perm);
  // the routing grid also ranks the assignments: the permute follows directly
  if ((s = do_route(c, L, ws, x, w_g, logit_bias, select_bias,
                    RouteOut{nullptr, idx, w, fo, Po, ao, cnt, kept, offsets, z_loss}, st)) !=
      MOE_OK)
    return s;
  // the permute kernel's extra blocks reduce the routing statistics
  const StatsArgs sa = make_stats(c, ws, L.status, route_grid(c, L), cnt, fo, Po, ao, z_loss);
  // top-1 bf16 layers without shared experts: the combine is fused into the
  // down-projection (and the permute writes the zero rows of dropped tokens)
  const bool fused_combine = c.dtype == MOE_BF16 && c.k == 1 && c.n_shared == 0;
  // MX FP8 experts: the permute writes the rows quantised, at padded offsets
  const bool mx = mx_experts(c);
  if ((s = launch_permute(c, idx, at<int32_t>(ws, L.crank), at<int32_t>(ws, L.hist), kept,
                          offsets, perm_token, slot_of, x, mx ? at<void>(ws, L.xq) : x_perm, st,
                          fused_combine ? out : nullptr, sa,
                          mx ? at<uint8_t>(ws, L.xq_sf) : nullptr, L.mx_rows / 128)) != MOE_OK)
    return s;
  FfnIn in{x_perm, w1, b1, w2, b2, x, ws1, wsb1, ws2, wsb2, offsets, mx};
  if (fused_combine) {
    const FfnScatter sc{out, perm_token, w};
    return do_ffn(c, L, ws, in, Y, Ys, st, &sc);
  }
  if ((s = do_ffn(c, L, ws, in, Y, Ys, st)) != MOE_OK) return s;
  return do_combine(c, Y, slot_of, w, c.n_shared > 0 ? Ys : nullptr, out, st);
}

moe_status moe_mxfp8_weight_bytes(int32_t G, int32_t N, int32_t K, size_t* bytes) {
  if (!bytes || G < 1 || N < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED;
  const size_t codes = static_cast<size_t>(G) * N * K;
  *bytes = codes + codes / 32 + mx_tile_records(G, N, K) * 4096;
  return MOE_OK;
}

moe_status moe_quantize_mxfp8(const void* w, int32_t G, int32_t N, int32_t K, int32_t glu,
                              void* packed, moe_stream stream) {
  size_t bytes = 0;
  moe_status s = moe_mxfp8_weight_bytes(G, N, K, &bytes);
  if (s != MOE_OK) return s;
  if (!w || !packed || (glu != 0 && glu != 1)) return MOE_ERR_INVALID_ARG;
  if (glu && N % 256 != 0) return MOE_ERR_UNSUPPORTED;   // two halves of whole 128-row tiles
  const int64_t rows = static_cast<int64_t>(G) * N;
  if (rows > static_cast<int64_t>(INT_MAX) * 8) return MOE_ERR_UNSUPPORTED;
  uint8_t* codes = static_cast<uint8_t*>(packed);
  uint8_t* sf = codes + static_cast<size_t>(G) * N * K;
  const int grid = static_cast<int>((rows + 7) / 8);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  k_quant_weights_mx<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w), G, N, K, glu,
                                           codes, sf);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  const int64_t recs = mx_tile_records(G, N, K);
  k_sf_tiles_mx<<<static_cast<unsigned>((recs * 256 + 255) / 256), 256, 0, st>>>(
      sf, recs, N / 128, (N + 255) / 256, sf + static_cast<size_t>(G) * N * K / 32);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_expert_capacity(const moe_config* cfg, int32_t* C) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!C) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  *C = expert_choice(c) ? ec_capacity(c) : (c.capacity_factor > 0.f ? capacity_of(c) : -1);
  return MOE_OK;
}

moe_status moe_route_expert_choice(const moe_config* cfg, const void* x, const void* w_g,
                                   const float* logit_bias, float* logits, int32_t* ec_token,
                                   float* ec_w, int32_t* ec_slot, float* f, float* P, float* aux,
                                   float* z_loss, void* ws, size_t ws_bytes, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(c);
  if ((s = check_ws(c, ws, ws_bytes, L)) != MOE_OK) return s;
  if (!f || !P || !aux) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    if (z_loss && cudaMemsetAsync(z_loss, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    return zero_stats(c, nullptr, f, P, aux, nullptr, nullptr, st);
  }
  if (!x || !w_g || !ec_slot) return MOE_ERR_INVALID_ARG;
  if (ec_capacity(c) > 0 && (!ec_token || !ec_w)) return MOE_ERR_INVALID_ARG;
  return do_route_ec(c, L, ws, x, w_g, logit_bias,
                     EcOut{logits, ec_token, ec_w, ec_slot, nullptr, at<int32_t>(ws, L.offsets),
                           nullptr, f, P, aux, z_loss},
                     st);
}

moe_status moe_permute_expert_choice(const moe_config* cfg, const void* x,
                                     const int32_t* ec_token, int32_t* offsets, void* x_perm,
                                     moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (ec_capacity(c) > 0 && (!x || !ec_token || !x_perm)) return MOE_ERR_INVALID_ARG;
  return do_permute_ec(c, x, ec_token, offsets, x_perm, st);
}

moe_status moe_combine_expert_choice(const moe_config* cfg, const void* y_perm,
                                     const int32_t* ec_slot, const float* ec_w,
                                     const void* y_shared, void* out, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!ec_slot || !out) return MOE_ERR_INVALID_ARG;
  if (ec_capacity(c) > 0 && (!y_perm || !ec_w)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
  return do_combine_ec(c, y_perm, ec_slot, ec_w, nullptr, c.n_shared > 0 ? y_shared : nullptr,
                       out, static_cast<cudaStream_t>(stream));
}

moe_status moe_check_status(void* ws, moe_stream stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  auto st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    return (v & DEV_ERR_BAD_EXPERT_INDEX) ? MOE_ERR_INVALID_ARG : MOE_ERR_TIMEOUT;
  }
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "a device-side bounded wait gave up";
  }
  return "unknown status";
}

}  // extern "C"
