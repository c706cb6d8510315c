/*
 * moe.h - C ABI of libmoe: the forward pass of a sparse Mixture-of-Experts FFN
 * layer on one NVIDIA B300 (sm_103a).
 *
 * The operation (notation of the pages this library restates):
 *   logits = x . W_g (+ logit_bias)                  router, no bias by default
 *   gate   : softmax over E -> top-k -> renormalise   ("SparseMoEGate")
 *          | top-k on logits -> softmax over the k    ("top_k_gating")
 *          | top-k on softmax + select_bias, weights from the unbiased
 *            softmax renormalised                     (DeepSeek-V3 bias)
 *   C      = max(floor(CF * T / E), min_capacity) when CF > 0; the assignments
 *            of an expert are ranked in ascending t*k + j and kept iff rank < C
 *   y      = sum_kept w[t,j] * FFN_{idx[t,j]}(x_t) + sum_s FFN_s(x_t)
 *   FFN(v) = act(v W1^T + b1) W2^T + b2, act = GELU_erf (default) or SiLU;
 *            SwiGLU: (SiLU(v W1g^T + b1g) * (v W1u^T + b1u)) W2^T + b2
 *   f_i, P_i, aux = alpha * E * sum_i f_i P_i          (Switch load balance)
 *   z      = mean_t logsumexp_e(logits[t, e])^2        (router z-loss)
 *   Expert Choice: C = min(max(floor(CF * T / E), min_capacity), T); expert e
 *            takes the C tokens with the largest logits[t, e] (lower t first
 *            on equal logits); y = sum over the experts e that took t of
 *            p[t, e] * FFN_e(x_t) + shared, p = softmax over the experts
 *
 * Sources: "混合专家大模型MoE架构选型与部署实践教程" §五 (SparseMoEGate,
 * SimpleMoELayer); "[BEE-30064] 混合專家架構與服務", 專家路由工作原理 (routing
 * steps 1-5, load_balance_loss); "AI-Research-SKILLs MoE 训练实战…全指南" §3.1,
 * §4.3, §6.1 (SiLU experts; SwiGLU named for Mixtral), §7.1, §8.2;
 * "第7章 Mixture of Experts" §7.1-§7.4.
 *
 * Conventions for every entry point
 *  - Ownership: the caller owns every buffer.  Unless stated otherwise a
 *    pointer is a DEVICE pointer on the current CUDA device.  The library never
 *    allocates device memory; scratch comes from the caller's workspace `ws`
 *    of at least moe_workspace_size() bytes, initialised once with
 *    moe_workspace_init().  A workspace serves one call at a time: calls that
 *    share one must be ordered (the same stream, or streams joined by
 *    events), since its header holds counters each call leaves at zero.
 *  - Execution: every call validates its arguments on the host first; on an
 *    error it returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE with NOTHING enqueued.  Otherwise it enqueues kernels on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and returns
 *    without synchronising.  MOE_ERR_CUDA reports a failed launch.
 *  - Device-side give-ups (a bounded wait inside a kernel that ran out) set a
 *    status word in `ws`; moe_check_status() synchronises and reports it.
 *  - Layouts are row-major.  Expert weights use nn.Linear's [out, in]
 *    (K-contiguous) layout.  W_g is [d_model, E].  Element type of x, W_g,
 *    expert weights/biases and the activations is cfg->dtype (fp32 or bf16);
 *    routing weights, logits, f, P and aux are always fp32, indices int32.
 *  - Determinism: outputs are bitwise reproducible run to run; no output is
 *    produced with floating-point atomics.
 *  - Dropped assignments have slot_of = -1 and contribute 0 to the output.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* moe_stream;   /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* bad pointer / size / enum value            */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. bf16 with d % 8 != 0) */
  MOE_ERR_WORKSPACE = 3,     /* ws NULL, too small or misaligned           */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed       */
  MOE_ERR_TIMEOUT = 5        /* a device-side bounded wait gave up         */
} moe_status;

typedef enum {
  MOE_ROUTE_SOFTMAX_TOPK = 0,    /* softmax over E, top-k, renormalise if cfg.renorm */
  MOE_ROUTE_TOPK_SOFTMAX = 1,    /* top-k on logits, softmax over the k              */
  MOE_ROUTE_BIASED_SOFTMAX = 2,  /* select on softmax + select_bias; weights = unbiased
                                    softmax renormalised over the k                  */
  MOE_ROUTE_EXPERT_CHOICE = 3    /* every expert takes its C tokens of largest logit;
                                    weight = the token's softmax probability; needs
                                    capacity_factor > 0; k is not used            */
} moe_route_kind;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  MOE_AUX_TOPK_COUNT = 0,   /* f_i = (#assignments to i) / T, sum f = k   */
  MOE_AUX_ARGMAX = 1        /* f_i = (#tokens whose largest logit is i) / T */
} moe_aux_f;

/* Storage of the expert weights w1, w2 (see moe_quantize_mxfp8). */
typedef enum {
  MOE_EXPERT_DENSE = 0,   /* in cfg.dtype                                       */
  MOE_EXPERT_MXFP8 = 1    /* MX FP8: e4m3 codes + one power-of-two scale per 32
                             elements along K, one packed buffer per tensor; the
                             activations are quantised the same way on the fly  */
} moe_expert_fmt;

typedef enum {
  MOE_ACT_GELU = 0,     /* GELU_erf(h), h = x W1^T + b1                       */
  MOE_ACT_SILU = 1,     /* h * sigmoid(h)                                     */
  MOE_ACT_SWIGLU = 2    /* W1 holds 2F rows: the gate projection's F rows, then
                           the up projection's F rows (b1 likewise 2F); the
                           hidden activation is SiLU(h_gate) * h_up, F wide  */
} moe_act;

/* The problem statement.  All fields are read by every entry point. */
typedef struct {
  int32_t T;               /* tokens, >= 0                                  */
  int32_t d_model;         /* d, > 0                                        */
  int32_t d_ff;            /* F, > 0                                        */
  int32_t E;               /* routed experts, 1..256                        */
  int32_t k;               /* experts per token, 1..min(E, 16)              */
  int32_t n_shared;        /* always-on shared experts, 0..4                */
  float capacity_factor;   /* CF; <= 0 means no capacity limit              */
  int32_t min_capacity;    /* lower bound on C when CF > 0, >= 0            */
  int32_t route;           /* moe_route_kind                                */
  int32_t renorm;          /* MOE_ROUTE_SOFTMAX_TOPK: 1 = renormalise over k */
  int32_t dtype;           /* moe_dtype                                     */
  int32_t has_bias;        /* 1: expert biases b1 [E,F], b2 [E,d] are given  */
  float aux_alpha;         /* alpha of the aux loss                         */
  int32_t aux_f;           /* moe_aux_f                                     */
  int32_t act;             /* moe_act: the experts' hidden activation        */
  int32_t y_f32;           /* 0: the expert outputs (y_perm, y_shared) are in
                              dtype; 1: they are fp32 (a bf16 layer then rounds
                              its expert outputs once, in the combine, instead
                              of twice).  Read by moe_grouped_ffn, moe_combine,
                              moe_combine_expert_choice and moe_forward.     */
  int32_t expert_fmt;      /* moe_expert_fmt.  MOE_EXPERT_MXFP8 needs dtype bf16,
                              top-k routing, n_shared = 0, and d_model and d_ff
                              multiples of 128 (else MOE_ERR_UNSUPPORTED).   */
} moe_config;

/* Bytes of workspace the entry points below need for `cfg` (host only). */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Clears the 1 MiB header of `ws` (stream-ordered): the device status word
 * and the counters and accumulators the kernels keep there, which must start
 * at zero and which every call leaves at zero again.  Call once after
 * allocating `ws`; ws_bytes must be >= 1 MiB (every moe_workspace_size is).
 * The header's layout does not depend on the configuration, so one
 * workspace may serve configurations of different sizes in turn. */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream stream);

/* Router + gating + load-balance statistics.
 *   x [T,d] dtype; w_g [d,E] dtype; logit_bias [E] fp32 or NULL (added to the
 *   logits); select_bias [E] fp32 or NULL (MOE_ROUTE_BIASED_SOFTMAX only).
 *   Outputs: logits [T,E] fp32 or NULL; topk_idx [T,k] int32 (descending
 *   selection score, lower expert index first on equal scores); topk_w [T,k]
 *   fp32; f [E], P [E] fp32; aux [1] fp32; z_loss [1] fp32 or NULL (the
 *   router z-loss of "AI-Research-SKILLs MoE 训练实战…全指南" §4.3: the mean over
 *   tokens of the squared log-sum-exp of the logits, logit_bias included).  f,
 *   P and z_loss count all T tokens before any capacity drop. */
moe_status moe_route(const moe_config* cfg, const void* x, const void* w_g,
                     const float* logit_bias, const float* select_bias,
                     float* logits, int32_t* topk_idx, float* topk_w,
                     float* f, float* P, float* aux, float* z_loss,
                     void* ws, size_t ws_bytes, moe_stream stream);

/* Dispatch: histogram, exclusive scan, capacity cut and row gather.
 *   topk_idx [T,k] int32 from moe_route.
 *   Outputs: counts [E] (assignments before the cut), kept [E] (= min(counts,
 *   C)), offsets [E+1] (exclusive scan of kept), perm_token [T*k] (token of
 *   each expert-ordered row; entries >= offsets[E] are unspecified), slot_of
 *   [T*k] (row of assignment t*k+j in x_perm, or -1 when dropped), x_perm
 *   [T*k, d] dtype (rows >= offsets[E] unspecified).
 *   An index outside [0, E), or one repeated in a token's row (after its
 *   first occurrence), drops that assignment (slot -1, not counted) and sets
 *   the status word: moe_check_status then returns MOE_ERR_INVALID_ARG. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       int32_t* counts, int32_t* kept, int32_t* offsets,
                       int32_t* perm_token, int32_t* slot_of, void* x_perm,
                       void* ws, size_t ws_bytes, moe_stream stream);

/* moe_permute without a workspace: the same dispatch (same kernels, same
 * outputs, bit for bit), with its scratch -- the in-chunk rank of each
 * assignment and the per-chunk expert counts -- held in a fixed array that
 * the library declares at file scope in device memory.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory themselves, e.g. a plugin living inside a host program that
 * owns every device allocation through its own pool, or code on a latency
 * path where a cudaMalloc (which may synchronise the device) is forbidden.
 *   Limits: T*k <= MOE_PERMUTE_NOALLOC_MAX_ASSIGNMENTS and
 *   32*ceil(ceil(T/32)/32)*E <= MOE_PERMUTE_NOALLOC_MAX_CHUNK_COUNTS (the
 *   per-chunk counts of each expert, rows padded to 32 chunks).  Larger sizes
 *   return MOE_ERR_UNSUPPORTED with nothing enqueued.
 *   Memory: every GPU that loads the library holds the array (8 MiB plus a
 *   2 KiB header) until the process exits.
 *   Set-up: every call looks up the array's device address on the current
 *   device; the first call on a device -- and the first after a device reset,
 *   which gives the array a new, undefined copy -- clears the header (a block
 *   counter and per-expert totals, which must start at zero) on `stream`;
 *   every call leaves them at zero again.  Make that first call before any
 *   stream capture.  No call allocates (no cudaMalloc, no cudaFree).
 *   Concurrency: all calls on one device share the one array, so calls whose
 *   kernels may overlap on the GPU (different streams without ordering) race
 *   and give wrong results; serialise them on one stream.
 *   Errors: as moe_permute, without ws.  An expert index outside [0, E) or
 *   repeated in a token's row drops that assignment (slot -1); unlike the
 *   workspace entry points, no status word reports it. */
#define MOE_PERMUTE_NOALLOC_MAX_ASSIGNMENTS 1048576
#define MOE_PERMUTE_NOALLOC_MAX_CHUNK_COUNTS 1048576
moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               int32_t* counts, int32_t* kept, int32_t* offsets,
                               int32_t* perm_token, int32_t* slot_of, void* x_perm,
                               moe_stream stream);

/* Expert MLPs as a grouped GEMM over the expert-contiguous rows.
 *   x_perm [T*k, d], offsets [E+1] (device; read on the device only).
 *   w1 [E,F1,d], b1 [E,F1] or NULL, w2 [E,d,F], b2 [E,d] or NULL, where
 *   F1 = 2F for MOE_ACT_SWIGLU (gate rows, then up rows) and F otherwise.
 *   Shared experts (cfg.n_shared > 0): x [T,d], ws1 [S,F1,d], wsb1 [S,F1] or
 *   NULL, ws2 [S,d,F], wsb2 [S,d] or NULL, output y_shared [S,T,d] dtype.
 *   Output y_perm [T*k, d]: row r = FFN_e(x_perm[r]) for the expert e
 *   whose range holds r; rows >= offsets[E] unspecified.  Both GEMMs
 *   accumulate in fp32; the hidden activation [rows, F] (in `ws`) is rounded
 *   once to dtype, the expert outputs y_perm and y_shared once to dtype, or
 *   stored in fp32 when cfg->y_f32 = 1. */
moe_status moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                           const void* w1, const void* b1, const void* w2, const void* b2,
                           const void* x, const void* ws1, const void* wsb1,
                           const void* ws2, const void* wsb2,
                           void* y_perm, void* y_shared,
                           void* ws, size_t ws_bytes, moe_stream stream);

/* Gate-weighted un-permute: out[t] = sum_{j: slot_of[t*k+j] >= 0}
 * topk_w[t,j] * y_perm[slot_of[t*k+j]] + sum_s y_shared[s,t], accumulated in
 * fp32 in ascending j then s, stored once in dtype.  y_perm [T*k, d] and
 * y_shared [S,T,d] are in dtype (fp32 when cfg->y_f32 = 1); y_shared may be
 * NULL when n_shared = 0. */
moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot_of,
                       const float* topk_w, const void* y_shared, void* out,
                       moe_stream stream);

/* MX FP8 expert weights ("AI-Research-SKILLs MoE 训练实战…全指南" §9.2 names FP8
 * serving of MoE layers; the format read here is the OCP Microscaling one):
 * every 32 consecutive elements of a weight row along K share a scale 2^s,
 * s = floor(log2(max |w|)) - 8 clamped to [-127, 127] (-127 for an all-zero
 * block), stored as the byte s + 127; each element is w / 2^s rounded to the
 * nearest e4m3 value (ties to even, saturating at +-448).
 *
 * moe_mxfp8_weight_bytes (host only): bytes of one packed tensor of G experts'
 * [N, K] weights: G*N*K code bytes, G*N*K/32 scale bytes, then
 * G*(K/128)*ceil(N/256) scale tile records of 4096 bytes.  N and K must be
 * multiples of 128.
 *
 * moe_quantize_mxfp8: packs bf16 weights w [G, N, K] (device) into `packed`
 * (device, moe_mxfp8_weight_bytes bytes), stream-ordered.  Codes: [G, N, K]
 * row-major.  Scales: 512-byte blocks, block (g, k / 128, n / 128) at
 * ((g * K/128 + k/128) * N/128 + n/128) * 512, the scale of row n and k-block
 * j = (k / 32) % 4 at byte 16 (n % 32) + 4 ((n % 128) / 32) + j of its block.
 * Tile records: record (g, k / 128, t) at ((g * K/128 + k/128) * ceil(N/256)
 * + t) * 4096 holds scale blocks (g, k / 128, 2t) and (g, k / 128, 2t + 1),
 * each four times in a row (the second all zeros when 2t + 1 = N/128): the
 * copy a 256-row tile of the CTA-pair GEMM loads in one piece.
 * glu = 1 packs a SwiGLU w1 ([2F, K]: gate rows, then up rows) with its rows
 * interleaved in 64-row halves -- packed row 128 t + i is gate row 64 t + i
 * for i < 64, up row F + 64 t + i - 64 otherwise -- which is the order the
 * layer reads; glu = 0 keeps the row order.  Pass the packed w1 / w2 to
 * moe_forward or moe_grouped_ffn with cfg.expert_fmt = MOE_EXPERT_MXFP8 (b1
 * and b2 stay in dtype, in their natural order). */
moe_status moe_mxfp8_weight_bytes(int32_t G, int32_t N, int32_t K, size_t* bytes);
moe_status moe_quantize_mxfp8(const void* w, int32_t G, int32_t N, int32_t K, int32_t glu,
                              void* packed, moe_stream stream);

/* Tokens per expert (host only): the capacity C of the configuration, or -1
 * when the top-k routing has no capacity limit (capacity_factor <= 0).  Under
 * MOE_ROUTE_EXPERT_CHOICE this is the number of tokens every expert takes. */
moe_status moe_expert_capacity(const moe_config* cfg, int32_t* C);

/* Expert Choice routing ("AI-Research-SKILLs MoE 训练实战…全指南" §4.2, "第7章
 * Mixture of Experts" §7.2): the router logits transposed to (experts, tokens)
 * and a top-C over the tokens of each expert, C = moe_expert_capacity().
 * cfg->route must be MOE_ROUTE_EXPERT_CHOICE.
 *   x [T,d] dtype; w_g [d,E] dtype; logit_bias [E] fp32 or NULL.
 *   Outputs: logits [T,E] fp32 or NULL; ec_token [E,C] int32 (the tokens
 *   expert e took, ascending); ec_w [E,C] fp32 (their gate weights p[t,e]);
 *   ec_slot [E,T] int32 (row e*C + r of x_perm holding token t for expert e,
 *   or -1); f [E] (= C/T with MOE_AUX_TOPK_COUNT), P [E], aux [1], z_loss [1]
 *   or NULL as in moe_route. */
moe_status moe_route_expert_choice(const moe_config* cfg, const void* x, const void* w_g,
                                   const float* logit_bias, float* logits,
                                   int32_t* ec_token, float* ec_w, int32_t* ec_slot,
                                   float* f, float* P, float* aux, float* z_loss,
                                   void* ws, size_t ws_bytes, moe_stream stream);

/* Expert Choice dispatch: x_perm [E*C, d] with row e*C + r = x[ec_token[e,r]],
 * and offsets [E+1] = e*C for moe_grouped_ffn. */
moe_status moe_permute_expert_choice(const moe_config* cfg, const void* x,
                                     const int32_t* ec_token, int32_t* offsets,
                                     void* x_perm, moe_stream stream);

/* Expert Choice combine: out[t] = sum over e ascending with ec_slot[e,t] >= 0
 * of ec_w[ec_slot[e,t]] * y_perm[ec_slot[e,t]] + sum_s y_shared[s,t],
 * accumulated in fp32 and stored once in dtype (0 plus the shared experts for
 * a token no expert took). */
moe_status moe_combine_expert_choice(const moe_config* cfg, const void* y_perm,
                                     const int32_t* ec_slot, const float* ec_w,
                                     const void* y_shared, void* out, moe_stream stream);

/* The whole layer: route -> permute -> grouped FFN -> combine, all stream
 * ordered with no host synchronisation.  Intermediates live in `ws`.  For a
 * bf16 top-1 layer without shared experts the combine is folded into the
 * down-projection (out[t] = w_t * FFN(x_t) rounded once to bf16, 0 for a
 * dropped token), which skips the rounding of the expert output that the
 * step-by-step entry points do.
 *   Outputs: out [T,d] dtype; topk_idx [T,k]; topk_w [T,k]; counts [E];
 *   f [E]; P [E]; aux [1]; z_loss [1] (as in moe_route).  Any of topk_idx ..
 *   z_loss may be NULL; out may not.  Under MOE_ROUTE_EXPERT_CHOICE topk_idx
 *   and topk_w receive ec_token [E,C] and ec_w [E,C] of
 *   moe_route_expert_choice, counts[e] = C, and select_bias is not used. */
moe_status moe_forward(const moe_config* cfg, const void* x, const void* w_g,
                       const float* logit_bias, const float* select_bias,
                       const void* w1, const void* b1, const void* w2, const void* b2,
                       const void* ws1, const void* wsb1, const void* ws2, const void* wsb2,
                       void* out, int32_t* topk_idx, float* topk_w, int32_t* counts,
                       float* f, float* P, float* aux, float* z_loss,
                       void* ws, size_t ws_bytes, moe_stream stream);

/* Synchronises `stream`, reads and clears the device status word of `ws`.
 * Returns MOE_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * check, MOE_ERR_CUDA if the stream reports an error, else MOE_OK. */
moe_status moe_check_status(void* ws, moe_stream stream);

/* Static string for a status code (host only). */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
