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

#include "moe.h"
#include "dispatch.cuh"
#include "gemm_tc.cuh"
#include "groups.cuh"
#include "route.cuh"

using namespace moe;

namespace {

// ---------------------------------------------------------------- config
constexpr int kTcRouterMinT = 256;     // bf16 routers with T below this use the FFMA kernel
constexpr size_t kAlign = 256;
// workspace header (64 bytes, zeroed by moe_workspace_init): the device status
// word at byte 0 and the finalize kernel's self-resetting block counter here
constexpr size_t kCounterOffset = 16;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int next_pow2_min16(int v) {
  int p = 16;
  while (p < v) p <<= 1;
  return p;
}

inline size_t elem_bytes(const moe_config& c) { return c.dtype == MOE_BF16 ? 2 : 4; }

moe_status validate(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model <= 0 || c->d_ff <= 0) return MOE_ERR_INVALID_ARG;
  if (c->E < 1 || c->E > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > c->E || c->k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > kMaxShared) return MOE_ERR_INVALID_ARG;
  if (c->min_capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->route < MOE_ROUTE_SOFTMAX_TOPK || c->route > MOE_ROUTE_BIASED_SOFTMAX)
    return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->aux_f != MOE_AUX_TOPK_COUNT && c->aux_f != MOE_AUX_ARGMAX) return MOE_ERR_INVALID_ARG;
  if (c->renorm != 0 && c->renorm != 1) return MOE_ERR_INVALID_ARG;
  if (c->has_bias != 0 && c->has_bias != 1) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->capacity_factor) || !std::isfinite(c->aux_alpha))
    return MOE_ERR_INVALID_ARG;
  const int64_t Tk = static_cast<int64_t>(c->T) * c->k;
  const int64_t rows_h = Tk + static_cast<int64_t>(c->n_shared) * c->T;
  if (rows_h > (INT_MAX / 2)) return MOE_ERR_INVALID_ARG;
  // 16-byte rows for vector loads and TMA strides
  if (c->d_model % 8 != 0 || c->d_ff % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_F32 && c->E > 64) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int capacity_of(const moe_config& c) {
  if (!(c.capacity_factor > 0.f)) return INT_MAX;
  const double v = std::floor(static_cast<double>(c.capacity_factor) * c.T / c.E);
  int cap = v > static_cast<double>(INT_MAX / 2) ? INT_MAX / 2 : static_cast<int>(v);
  return std::max(cap, c.min_capacity);
}

bool use_tc_router(const moe_config& c) {
  return c.dtype == MOE_BF16 && (c.E > 64 || c.T >= kTcRouterMinT);
}

struct Layout {
  size_t status, logits, wgT, p_part, c_part, a_part, rank;
  size_t idx, w, counts, kept, offsets, perm_token, slot_of, fin, f, P, aux;
  size_t x_perm, H, Y, Ys, total;
  int nb, E_pad;
  bool tc_router;
};

Layout make_layout(const moe_config& c) {
  Layout L{};
  const size_t T = c.T, E = c.E, k = c.k, S = c.n_shared, d = c.d_model, F = c.d_ff;
  const size_t eb = elem_bytes(c);
  L.nb = route_blocks(c.T);
  L.E_pad = next_pow2_min16(c.E);
  L.tc_router = use_tc_router(c);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + std::max<size_t>(bytes, 1), kAlign);
    return at;
  };
  L.status = take(64);
  L.logits = take(L.tc_router ? T * L.E_pad * 4 : 0);
  L.wgT = take(L.tc_router ? static_cast<size_t>(L.E_pad) * d * 2 : 0);
  L.p_part = take(static_cast<size_t>(L.nb) * E * 4);
  L.c_part = take(static_cast<size_t>(L.nb) * E * 4);
  L.a_part = take(static_cast<size_t>(L.nb) * E * 4);
  L.rank = take(T * k * 4);
  L.idx = take(T * k * 4);
  L.w = take(T * k * 4);
  L.counts = take(E * 4);
  L.kept = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm_token = take(T * k * 4);
  L.slot_of = take(T * k * 4);
  L.fin = take(E * 8);
  L.f = take(E * 4);
  L.P = take(E * 4);
  L.aux = take(4);
  L.x_perm = take(T * k * d * eb);
  L.H = take((T * k + S * T) * F * eb);
  L.Y = take(T * k * d * 4);
  L.Ys = take(S * T * d * 4);
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

inline moe_status launch_ok() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
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

// ---------------------------------------------------------------- GEMM launch
template <int BN, int STAGES, int EPI>
moe_status launch_tc_inst(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                          const CUtensorMap& b1, const TcArgs& args, int64_t row_tiles_ub,
                          cudaStream_t st) {
  constexpr size_t smem = TcSmem<BN, STAGES>::bytes();
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(k_gemm_tc<BN, STAGES, EPI>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t n_tiles = (args.N + BN - 1) / BN;
  const int64_t ub = std::max<int64_t>(1, row_tiles_ub * n_tiles);
  const int grid = static_cast<int>(std::min<int64_t>(ub, num_sms()));
  k_gemm_tc<BN, STAGES, EPI><<<grid, 192, smem, st>>>(a0, a1, b0, b1, args);
  return launch_ok();
}

int pick_bn_small(int N) { return N >= 64 ? 64 : 64; }

// Row tiles (128 rows) of a grouped GEMM over n_rows expert-ordered rows in
// E groups, estimated on the host: the per-expert counts stay on the device.
int64_t est_row_tiles(int64_t n_rows, int E) {
  const int64_t dense = (n_rows + 127) / 128 + E / 2;    // plus ragged group tails
  return std::max<int64_t>(dense, std::min<int64_t>(E, n_rows));
}

// Tile width for a weight-streaming grouped GEMM: the persistent grid runs
// ceil(tiles / SMs) rounds, each as long as one tile, whose cost grows with
// BN (the B slab) plus a fixed share for A and the epilogue.  Picks the BN
// with the smallest estimated makespan, preferring the wider tile on ties.
int pick_bn_waves(int N, int64_t row_tiles, int sms) {
  int best = 256;
  int64_t best_cost = INT64_MAX;
  for (int bn : {256, 128}) {
    const int64_t tiles = row_tiles * ((N + bn - 1) / bn);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const int64_t cost = rounds * (bn + 64);
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return N < 128 ? pick_bn_small(N) : best;
}

int pick_bn(int N, bool allow_small) {
  if (N >= 256) return 256;
  if (N >= 128) return 128;
  if (N >= 64 || !allow_small) return 64;
  if (N >= 32) return 32;
  return 16;
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
  } else if (epi == EPI_BIAS_F32) {
    switch (BN) {
      case 64: return launch_tc_inst<64, 8, EPI_BIAS_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 128: return launch_tc_inst<128, 6, EPI_BIAS_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 256: return launch_tc_inst<256, 4, EPI_BIAS_F32>(a0, a1, b0, b1, args, row_tiles_ub, st);
    }
  } else if (epi == EPI_GELU_BF16) {
    switch (BN) {
      case 64: return launch_tc_inst<64, 8, EPI_GELU_BF16>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 128: return launch_tc_inst<128, 6, EPI_GELU_BF16>(a0, a1, b0, b1, args, row_tiles_ub, st);
      case 256: return launch_tc_inst<256, 4, EPI_GELU_BF16>(a0, a1, b0, b1, args, row_tiles_ub, st);
    }
  }
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
};

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
  ra.p_part = at<float>(ws, L.p_part);
  ra.c_part = at<int32_t>(ws, L.c_part);
  ra.a_part = at<int32_t>(ws, L.a_part);
  const int nb = L.nb;
  moe_status s = MOE_OK;
  if (L.tc_router) {
    __nv_bfloat16* wgT = at<__nv_bfloat16>(ws, L.wgT);
    float* logits_ws = at<float>(ws, L.logits);
    dim3 tgrid((c.d_model + 31) / 32, (L.E_pad + 31) / 32);
    k_transpose_wg<<<tgrid, dim3(32, 8), 0, st>>>(static_cast<const __nv_bfloat16*>(w_g),
                                                   c.d_model, c.E, L.E_pad, wgT);
    if ((s = launch_ok()) != MOE_OK) return s;
    CUtensorMap ma, mb;
    if (!map_a(&ma, x, c.d_model, c.T) || !map_b(&mb, wgT, c.d_model, L.E_pad, 1, L.E_pad))
      return MOE_ERR_CUDA;
    TcArgs ta{};
    ta.gs = GroupSpec{nullptr, 1, c.T, 0, 0, 0, 0, 0, 0};
    ta.N = L.E_pad;
    ta.K = c.d_model;
    ta.out = logits_ws;
    ta.out1 = logits_ws;
    ta.ldo = L.E_pad;
    ta.err = at<int>(ws, L.status);
    s = launch_tc(EPI_F32, ma, ma, mb, mb, ta, L.E_pad, (c.T + 127) / 128 + 1, st);
    if (s != MOE_OK) return s;
    ra.logits_in = logits_ws;
    ra.ld_in = L.E_pad;
    if (c.E <= 32) k_gate<1><<<nb, kRouteWarps * 32, 0, st>>>(ra);
    else if (c.E <= 64) k_gate<2><<<nb, kRouteWarps * 32, 0, st>>>(ra);
    else if (c.E <= 128) k_gate<4><<<nb, kRouteWarps * 32, 0, st>>>(ra);
    else k_gate<8><<<nb, kRouteWarps * 32, 0, st>>>(ra);
  } else if (c.dtype == MOE_BF16) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* wb = static_cast<const __nv_bfloat16*>(w_g);
    if (c.E <= 8) k_route_warp<__nv_bfloat16, 8><<<nb, kRouteWarps * 32, 0, st>>>(ra, xb, wb);
    else if (c.E <= 16) k_route_warp<__nv_bfloat16, 16><<<nb, kRouteWarps * 32, 0, st>>>(ra, xb, wb);
    else if (c.E <= 32) k_route_warp<__nv_bfloat16, 32><<<nb, kRouteWarps * 32, 0, st>>>(ra, xb, wb);
    else k_route_warp<__nv_bfloat16, 64><<<nb, kRouteWarps * 32, 0, st>>>(ra, xb, wb);
  } else {
    const auto* xf = static_cast<const float*>(x);
    const auto* wf = static_cast<const float*>(w_g);
    if (c.E <= 8) k_route_warp<float, 8><<<nb, kRouteWarps * 32, 0, st>>>(ra, xf, wf);
    else if (c.E <= 16) k_route_warp<float, 16><<<nb, kRouteWarps * 32, 0, st>>>(ra, xf, wf);
    else if (c.E <= 32) k_route_warp<float, 32><<<nb, kRouteWarps * 32, 0, st>>>(ra, xf, wf);
    else k_route_warp<float, 64><<<nb, kRouteWarps * 32, 0, st>>>(ra, xf, wf);
  }
  if ((s = launch_ok()) != MOE_OK) return s;
  k_route_finalize<<<c.E, 256, 0, st>>>(nb, c.T, c.E, c.aux_f, c.aux_alpha, ra.p_part,
                                         ra.c_part, ra.a_part, o.f, o.P, o.aux,
                                         at<double>(ws, L.fin),
                                         at<unsigned int>(ws, L.status + kCounterOffset));
  return launch_ok();
}

int kmax_of(int k) { return k <= 2 ? 2 : (k <= 4 ? 4 : (k <= 8 ? 8 : 16)); }

moe_status do_permute(const moe_config& c, const Layout& L, void* ws, const void* x,
                      const int32_t* idx, int32_t* counts, int32_t* kept, int32_t* offsets,
                      int32_t* perm_token, int32_t* slot_of, void* x_perm, cudaStream_t st) {
  int32_t* rank = at<int32_t>(ws, L.rank);
  const int Tk = c.T * c.k;
  k_rank<<<c.E, 1024, 0, st>>>(idx, Tk, capacity_of(c), rank, counts, kept);
  moe_status s;
  if ((s = launch_ok()) != MOE_OK) return s;
  const int row_bytes = c.d_model * static_cast<int>(elem_bytes(c));
  const int grid = std::max(1, std::min((c.T + 7) / 8, num_sms() * 8));
  const auto* xb = static_cast<const uint8_t*>(x);
  auto* xp = static_cast<uint8_t*>(x_perm);
  switch (kmax_of(c.k)) {
    case 2: k_permute<2><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
    case 4: k_permute<4><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
    case 8: k_permute<8><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
    default: k_permute<16><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
  }
  return launch_ok();
}

// ---------------------------------------------------------------- fixed scratch
// Rank array of moe_permute_noalloc: a file-scope device array, so that entry
// point needs no caller workspace and allocates nothing.  Host code must not
// pass `g_noalloc_rank` itself to a kernel (in host code the name is only a
// host-side stand-in): the device address comes from cudaGetSymbolAddress,
// looked up once per device with that device current.
constexpr int64_t kNoallocRankEntries = MOE_PERMUTE_NOALLOC_MAX_ASSIGNMENTS;
static __device__ __align__(256) int32_t g_noalloc_rank[kNoallocRankEntries];

// Device address of g_noalloc_rank on the current device, or null when the
// lookup fails.  The first call on each device does the lookup.
int32_t* noalloc_rank_address() {
  constexpr int kMaxDevices = 64;
  static int32_t* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_rank) != cudaSuccess || !p) return nullptr;
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
}

// The dispatch of do_permute with the rank scratch passed in directly.
moe_status permute_with_rank(const moe_config& c, int32_t* rank, const void* x,
                             const int32_t* idx, int32_t* counts, int32_t* kept,
                             int32_t* offsets, int32_t* perm_token, int32_t* slot_of,
                             void* x_perm, cudaStream_t st) {
  const int Tk = c.T * c.k;
  k_rank<<<c.E, 1024, 0, st>>>(idx, Tk, capacity_of(c), rank, counts, kept);
  moe_status s;
  if ((s = launch_ok()) != MOE_OK) return s;
  const int row_bytes = c.d_model * static_cast<int>(elem_bytes(c));
  const int grid = std::max(1, std::min((c.T + 7) / 8, num_sms() * 8));
  const auto* xb = static_cast<const uint8_t*>(x);
  auto* xp = static_cast<uint8_t*>(x_perm);
  switch (kmax_of(c.k)) {
    case 2: k_permute<2><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
    case 4: k_permute<4><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
    case 8: k_permute<8><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
    default: k_permute<16><<<grid, 256, 0, st>>>(idx, rank, kept, c.T, c.k, c.E, row_bytes, xb, xp, offsets, perm_token, slot_of); break;
  }
  return launch_ok();
}

struct FfnIn {
  const void *x_perm, *w1, *b1, *w2, *b2, *x, *ws1, *wsb1, *ws2, *wsb2;
  const int32_t* offsets;
};

moe_status do_ffn(const moe_config& c, const Layout& L, void* ws, const FfnIn& in, void* y_perm,
                  void* y_shared, cudaStream_t st) {
  const int64_t T = c.T, Tk = static_cast<int64_t>(c.T) * c.k, S = c.n_shared;
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
  if (c.dtype == MOE_BF16) {
    CUtensorMap ma0, ma1, mb0, mb1;
    // up-projection + GELU:  H = GELU(x_perm W1^T + b1)
    if (!map_a(&ma0, in.x_perm, d, std::max<int64_t>(Tk, 1))) return MOE_ERR_CUDA;
    const int64_t rt = est_row_tiles(Tk, c.E) + S * ((T + 127) / 128);
    const int bn_up = pick_bn_waves(F, rt, num_sms());
    if (!map_b(&mb0, in.w1, d, F, c.E, bn_up)) return MOE_ERR_CUDA;
    if (S > 0) {
      if (!map_a(&ma1, in.x, d, T) || !map_b(&mb1, in.ws1, d, F, S, bn_up)) return MOE_ERR_CUDA;
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
    up.bias0 = static_cast<const __nv_bfloat16*>(b1);
    up.bias1 = static_cast<const __nv_bfloat16*>(wsb1);
    up.err = at<int>(ws, L.status);
    if ((s = launch_tc(EPI_GELU_BF16, ma0, ma1, mb0, mb1, up, bn_up, row_tiles_ub, st)) != MOE_OK)
      return s;
    // down-projection:  y = H W2^T + b2
    CUtensorMap ha, hb0, hb1;
    if (!map_a(&ha, H, F, Tk + S * T)) return MOE_ERR_CUDA;
    const int bn_dn = pick_bn_waves(d, rt, num_sms());
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
    return launch_tc(EPI_BIAS_F32, ha, ha, hb0, hb1, dn, bn_dn, row_tiles_ub, st);
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
  up.gelu = 1;
  int grid = static_cast<int>(std::min<int64_t>(tiles_ub * ((F + 63) / 64), num_sms() * 4));
  k_gemm_simt_f32<<<std::max(grid, 1), 256, 0, st>>>(up);
  if ((s = launch_ok()) != MOE_OK) return s;
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
  dn.gelu = 0;
  grid = static_cast<int>(std::min<int64_t>(tiles_ub * ((d + 63) / 64), num_sms() * 4));
  k_gemm_simt_f32<<<std::max(grid, 1), 256, 0, st>>>(dn);
  return launch_ok();
}

moe_status do_combine(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                      const float* w, const void* y_shared, void* out, cudaStream_t st) {
  const int grid = std::max(1, std::min((c.T + 7) / 8, num_sms() * 8));
  const int S = y_shared ? c.n_shared : 0;
#define MOE_COMBINE(TE, KM)                                                                  \
  k_combine<TE, KM><<<grid, 256, 0, st>>>(static_cast<const float*>(y_perm), slot_of, w,   \
                                          static_cast<const float*>(y_shared), S, c.T, c.k, \
                                          c.d_model, static_cast<TE*>(out))
  const int km = kmax_of(c.k);
  if (c.dtype == MOE_BF16) {
    if (km == 2) MOE_COMBINE(__nv_bfloat16, 2);
    else if (km == 4) MOE_COMBINE(__nv_bfloat16, 4);
    else if (km == 8) MOE_COMBINE(__nv_bfloat16, 8);
    else MOE_COMBINE(__nv_bfloat16, 16);
  } else {
    if (km == 2) MOE_COMBINE(float, 2);
    else if (km == 4) MOE_COMBINE(float, 4);
    else if (km == 8) MOE_COMBINE(float, 8);
    else MOE_COMBINE(float, 16);
  }
#undef MOE_COMBINE
  return launch_ok();
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
  if (!ws || ws_bytes < 64 || reinterpret_cast<uintptr_t>(ws) % kAlign != 0)
    return MOE_ERR_WORKSPACE;
  return cudaMemsetAsync(ws, 0, 64, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* w_g,
                     const float* logit_bias, const float* select_bias, float* logits,
                     int32_t* topk_idx, float* topk_w, float* f, float* P, float* aux, void* ws,
                     size_t ws_bytes, moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if ((s = check_ws(c, ws, ws_bytes, L)) != MOE_OK) return s;
  if (!f || !P || !aux) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return zero_stats(c, nullptr, f, P, aux, nullptr, nullptr, st);
  if (!x || !w_g || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  return do_route(c, L, ws, x, w_g, logit_bias, select_bias,
                  RouteOut{logits, topk_idx, topk_w, f, P, aux}, st);
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
  if (!counts || !kept || !offsets) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return zero_stats(c, counts, nullptr, nullptr, nullptr, offsets, kept, st);
  if (!x || !topk_idx || !perm_token || !slot_of || !x_perm) return MOE_ERR_INVALID_ARG;
  return do_permute(c, L, ws, x, topk_idx, counts, kept, offsets, perm_token, slot_of, x_perm,
                    st);
}

moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               int32_t* counts, int32_t* kept, int32_t* offsets,
                               int32_t* perm_token, int32_t* slot_of, void* x_perm,
                               moe_stream stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (static_cast<int64_t>(c.T) * c.k > kNoallocRankEntries) return MOE_ERR_UNSUPPORTED;
  if (!counts || !kept || !offsets) return MOE_ERR_INVALID_ARG;
  auto st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return zero_stats(c, counts, nullptr, nullptr, nullptr, offsets, kept, st);
  if (!x || !topk_idx || !perm_token || !slot_of || !x_perm) return MOE_ERR_INVALID_ARG;
  int32_t* rank = noalloc_rank_address();
  if (!rank) return MOE_ERR_CUDA;
  return permute_with_rank(c, rank, x, topk_idx, counts, kept, offsets, perm_token, slot_of,
                           x_perm, st);
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
                       float* aux, void* ws, size_t ws_bytes, moe_stream stream) {
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
  if (c.T == 0) return zero_stats(c, counts, f, P, aux, nullptr, nullptr, st);
  if (!x || !w_g || !w1 || !w2) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (!ws1 || !ws2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && c.has_bias && (!wsb1 || !wsb2)) return MOE_ERR_INVALID_ARG;

  if ((s = do_route(c, L, ws, x, w_g, logit_bias, select_bias,
                    RouteOut{nullptr, idx, w, fo, Po, ao}, st)) != MOE_OK)
    return s;
  int32_t* kept = at<int32_t>(ws, L.kept);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* slot_of = at<int32_t>(ws, L.slot_of);
  void* x_perm = at<uint8_t>(ws, L.x_perm);
  if ((s = do_permute(c, L, ws, x, idx, cnt, kept, offsets, at<int32_t>(ws, L.perm_token),
                      slot_of, x_perm, st)) != MOE_OK)
    return s;
  void* Y = at<uint8_t>(ws, L.Y);
  void* Ys = at<uint8_t>(ws, L.Ys);
  FfnIn in{x_perm, w1, b1, w2, b2, x, ws1, wsb1, ws2, wsb2, offsets};
  if ((s = do_ffn(c, L, ws, in, Y, Ys, st)) != MOE_OK) return s;
  return do_combine(c, Y, slot_of, w, c.n_shared > 0 ? Ys : nullptr, out, st);
}

moe_status moe_check_status(void* ws, moe_stream stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  auto st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_TIMEOUT;
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
