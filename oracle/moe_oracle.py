"""Plain CPU oracle for the forward pass of a sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, constants or helpers with the
CUDA path: it is numpy in float64, one library primitive per step (a matmul, a
stable sort, ``erf``), with no blocking, fusion or reordering beyond what the
definitions below state.

Sources (page title, then section / listing / formula):

* [BAIDU]  "混合专家大模型MoE架构选型与部署实践教程", §五 "通用伪代码与门控配置示例":
  the ``SparseMoEGate`` router (linear without bias -> softmax -> top-k ->
  renormalise over the k; the aux loss as alpha * E * sum(f_i * P_i) with
  f_i = mean over tokens of the one-hot top-k mask) and ``SimpleMoELayer``
  (per-expert token lists, Linear -> GELU -> Linear experts, gate-weighted
  ``index_add_`` combine).  §七.1 for "overflow tokens are dropped or skip
  through the residual path".
* [BEE]    "[BEE-30064] 混合專家架構與服務", section "專家路由工作原理": the
  five routing steps (h = x @ W_g with W_g of shape [d_model, E]; top-k on h;
  softmax over only the chosen k; dispatch; weighted sum) and
  ``load_balance_loss`` (f_i from argmax one-hot routing, P_i = mean softmax,
  alpha * E * sum(f * P)).
* [SKILLS] "AI-Research-SKILLs MoE 训练实战…全指南": §3.1 ``MoELayer`` (softmax
  -> top-k -> renormalise), §4.3 ``load_balancing_loss`` (bincount of the
  chosen indices), ``router_z_loss`` and the DeepSeek-V3 bias remark, §7.1 ``DeepSeekMoE``
  (shared experts always computed and added with weight one), §8.2 the
  capacity formula ``int((tokens / num_experts) * capacity_factor)``.
  §6.1 ``MixtralMoEBlock`` (experts Linear -> SiLU -> Linear without bias,
  and the text naming SwiGLU as Mixtral's FFN activation).  §4.2 Expert
  Choice routing: the router's scores transposed to (experts, tokens) and a
  top-k over the tokens of each expert, k = its capacity.
* [CH7]    "第7章 Mixture of Experts": §7.1 MoE(x) = sum_i G(x)_i * E_i(x);
  §7.2 ``top_k_gating`` (top-k on logits, softmax over the k) and Expert
  Choice (each expert takes its top-C tokens, so every expert processes the
  same number; a token may be taken by several experts or by none); §7.3 shared +
  fine-grained experts; §7.4 the balance loss N * sum f_i p_i and capacity
  C = CF * n / N with ``int(...)``.

Readings where the pages are silent or disagree are stated at each function
(R-numbers match the readings table of the design notes).  Every function here
is pinned by ``tests/test_oracle_pins.py``; none is "parity unpinned".
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np
from scipy.special import erf, expit

ROUTE_SOFTMAX_TOPK = "softmax_topk"      # [BAIDU] SparseMoEGate, [SKILLS] §3.1
ROUTE_TOPK_SOFTMAX = "topk_softmax"      # [BEE] steps 2-3, [CH7] §7.2 top_k_gating
ROUTE_BIASED_SOFTMAX = "biased_softmax"  # [SKILLS] §4.3 / §7.1 DeepSeek-V3 bias
ROUTE_EXPERT_CHOICE = "expert_choice"    # [SKILLS] §4.2, [CH7] §7.2 Expert Choice (R19)
AUX_TOPK_COUNT = "topk_count"            # [BAIDU] one-hot of the top-k, summed
AUX_ARGMAX = "argmax"                    # [BEE] load_balance_loss, argmax routing
ACT_GELU = "gelu"                        # [BAIDU] §五, [SKILLS] §3.1 nn.GELU()
ACT_SILU = "silu"                        # [SKILLS] §6.1 MixtralMoEBlock nn.SiLU()
ACT_SWIGLU = "swiglu"                    # [SKILLS] §6.1 "SwiGLU" (R18)


@dataclass
class OracleConfig:
    """Problem statement: T tokens, d_model, d_ff, E routed experts, top-k,
    capacity factor, routing variant (the quantities [BAIDU] step one and the
    [CH7] symbol table name)."""

    T: int
    d_model: int
    d_ff: int
    E: int
    k: int
    n_shared: int = 0
    capacity_factor: float = 0.0   # <= 0 means no capacity limit
    min_capacity: int = 0
    route: str = ROUTE_SOFTMAX_TOPK
    renorm: bool = True
    aux_alpha: float = 0.01
    aux_f: str = AUX_TOPK_COUNT
    act: str = ACT_GELU
    experts: str = "dense"          # "dense" or "mxfp8" (R22: MX FP8 expert operands)


# --------------------------------------------------------------------------
# Step 1: router linear layer.  [BEE] step 1 (h = x @ W_g, W_g [d_model, E],
# "a single linear layer without bias"); [BAIDU] gate_proj(bias=False).
# --------------------------------------------------------------------------
def router_logits(x: np.ndarray, w_g: np.ndarray,
                  logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """logits = x @ W_g, accumulated in float64 and stored as float32.

    The logits are float32 quantities on both sides of the comparison; the
    product is exact in float64 for bf16 operands up to the final rounding.
    ``logit_bias`` (float32, [E]) is a fixed per-expert offset added to the
    float32 logits in float32 (the [SKILLS] §3.1 ``nn.Linear`` with bias, used
    here for the skewed decode workload).
    """
    h = (np.asarray(x, np.float64) @ np.asarray(w_g, np.float64)).astype(np.float32)
    if logit_bias is not None:
        h = (h + np.asarray(logit_bias, np.float32)).astype(np.float32)
    return h


def softmax(logits: np.ndarray) -> np.ndarray:
    """Row softmax in float64, max-subtracted (the value is the textbook
    exp(l_i) / sum_j exp(l_j))."""
    l = np.asarray(logits, np.float64)
    z = np.exp(l - l.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def select_topk(score: np.ndarray, k: int):
    """Top-k per row: descending score, the lower expert index first on equal
    scores (R4: the pages leave torch.topk's tie order open).

    Returns (idx [T,k] int64, margin [T]) where margin is the smallest gap
    between neighbours among the k+1 best scores (inf when k == E): a token
    whose margin is below the comparison threshold may legitimately be ordered
    differently by another summation order (R5).
    """
    s = np.asarray(score, np.float64)
    # a stable sort on -score keeps equal scores in ascending index order
    order = np.argsort(-s, axis=-1, kind="stable")
    idx = order[:, :k]
    E = s.shape[1]
    m = min(k + 1, E)
    top = np.take_along_axis(s, order[:, :m], axis=-1)
    if m >= 2:
        margin = np.min(top[:, :-1] - top[:, 1:], axis=-1)
    else:
        margin = np.full(s.shape[0], np.inf)
    return idx, margin


@dataclass
class GateResult:
    idx: np.ndarray       # [T,k] int64 expert ids
    w: np.ndarray         # [T,k] float64 gate weights
    p: np.ndarray         # [T,E] float64 unbiased softmax of the logits
    margin: np.ndarray    # [T] selection-score margin (see select_topk)
    score: Optional[np.ndarray] = None   # [T,E] float64 selection score (p, l or p + b)


def gate(logits: np.ndarray, cfg: OracleConfig,
         select_bias: Optional[np.ndarray] = None,
         idx_override: Optional[dict] = None) -> GateResult:
    """Gating in the three forms the pages give.

    * softmax_topk  ([BAIDU] gate steps 1-2, [SKILLS] §3.1, §6.1): p = softmax(l)
      over all E; choose the k largest p; w = p_sel / sum(p_sel) when renorm,
      else w = p_sel (the Switch top-1 gate value, reading R3).
    * topk_softmax  ([BEE] steps 2-3, [CH7] §7.2): choose the k largest logits;
      w = softmax over those k logits only.
    * biased_softmax ([SKILLS] §4.3 last paragraph, §7.1; DeepSeek-V3): choose
      the k largest p + select_bias; w = p_sel / sum(p_sel) from the unbiased
      p (reading R10: the bias is added to the probabilities and steers
      selection only).

    ``idx_override`` maps a token to an index row to use instead of the
    oracle's own choice (used for near-tie tokens, R5); weights are then
    recomputed from the oracle's own p / l for those indices.
    """
    l = np.asarray(logits, np.float32)
    p = softmax(l)
    if cfg.route == ROUTE_SOFTMAX_TOPK:
        score = p
    elif cfg.route == ROUTE_TOPK_SOFTMAX:
        score = l.astype(np.float64)
    elif cfg.route == ROUTE_BIASED_SOFTMAX:
        b = np.zeros(cfg.E) if select_bias is None else np.asarray(select_bias, np.float64)
        score = p + b[None, :]
    else:
        raise ValueError(cfg.route)
    idx, margin = select_topk(score, cfg.k)
    if idx_override:
        idx = idx.copy()
        for t, row in idx_override.items():
            idx[t] = np.asarray(row, dtype=idx.dtype)

    if cfg.route == ROUTE_TOPK_SOFTMAX:
        sel = np.take_along_axis(l.astype(np.float64), idx, axis=-1)
        z = np.exp(sel - sel.max(axis=-1, keepdims=True))
        w = z / z.sum(axis=-1, keepdims=True)
    else:
        sel = np.take_along_axis(p, idx, axis=-1)
        if cfg.route == ROUTE_BIASED_SOFTMAX or cfg.renorm:
            w = sel / sel.sum(axis=-1, keepdims=True)   # R16: sum >= max p > 0
        else:
            w = sel
    return GateResult(idx=idx, w=w, p=p, margin=margin, score=score)


# --------------------------------------------------------------------------
# Capacity and dispatch.  [SKILLS] §8.2 int((T / E) * CF); [CH7] §7.4
# capacity = int(capacity_factor * num_tokens / num_experts), overflow dropped.
# --------------------------------------------------------------------------
def capacity(cfg: OracleConfig) -> Optional[int]:
    """Tokens one expert may take, or None for no limit.

    C = floor(CF * T / E) (``int()`` of a positive float is floor), raised to
    ``min_capacity`` ([SKILLS] §5.1 min_capacity).  CF <= 0 means no limit.
    """
    if cfg.capacity_factor <= 0:
        return None
    c = int(math.floor(cfg.capacity_factor * cfg.T / cfg.E))
    return max(c, cfg.min_capacity)


@dataclass
class Dispatch:
    counts: np.ndarray      # [E] assignments per expert before the capacity cut
    kept: np.ndarray        # [E] min(counts, C)
    offsets: np.ndarray     # [E+1] exclusive prefix sum of kept
    perm_token: np.ndarray  # [sum kept] token of each expert-ordered row
    slot_of: np.ndarray     # [T*k] row of assignment t*k+j, -1 when dropped
    rank: np.ndarray        # [T*k] position of the assignment inside its expert


def dispatch(idx: np.ndarray, E: int, C: Optional[int]) -> Dispatch:
    """Group the (token, slot) assignments by expert.

    [BAIDU] SimpleMoELayer gathers, per expert, the tokens whose top-k row
    contains it (``torch.where``) in ascending token order; for several slots
    of one token the flat order t*k + j is used (R6).  An assignment is kept iff
    its rank within its expert is below C; dropped ones contribute nothing
    (reading R7: the layer outputs 0 for them, the residual add is the
    caller's).
    """
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")          # by expert, then by t*k+j
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    rank = np.empty(T * k, np.int64)
    rank[order] = np.arange(T * k) - starts[flat[order]]
    kept = counts if C is None else np.minimum(counts, C)
    offsets = np.concatenate([[0], np.cumsum(kept)]).astype(np.int64)
    keep = rank < (kept[flat])
    slot_of = np.where(keep, offsets[flat] + rank, -1).astype(np.int64)
    perm_token = np.empty(int(offsets[-1]), np.int64)
    perm_token[slot_of[keep]] = np.nonzero(keep)[0] // k
    return Dispatch(counts=counts, kept=kept.astype(np.int64), offsets=offsets,
                    perm_token=perm_token, slot_of=slot_of, rank=rank)


# --------------------------------------------------------------------------
# Expert Choice.  [SKILLS] §4.2: expert_scores = router(x) transposed to
# (experts, tokens), then topk over the tokens with k = the capacity per
# expert; [CH7] §7.2: each expert takes the Top-C tokens most related to it.
# --------------------------------------------------------------------------
@dataclass
class ExpertChoice:
    C: int                  # tokens per expert
    tokens: np.ndarray      # [E, C] int64 chosen tokens of each expert, ascending
    w: np.ndarray           # [E, C] float64 gate weight p[token, e]
    p: np.ndarray           # [T, E] float64 softmax of the logits over experts
    margin: np.ndarray      # [E] C-th minus (C+1)-th largest logit of the expert


def expert_choice_capacity(cfg: OracleConfig) -> int:
    """C = the top-k capacity C of ``capacity`` (floor(CF * T / E), raised to
    min_capacity), at most T.  Expert Choice needs CF > 0 (R19)."""
    C = capacity(cfg)
    if C is None:
        raise ValueError("Expert Choice routing needs a capacity factor > 0")
    return min(C, cfg.T)


def expert_choice(logits: np.ndarray, C: int,
                  override: Optional[dict] = None) -> ExpertChoice:
    """Each expert e takes the C tokens with the largest logit l[t, e] of its
    column, the lower token index first among equal logits (R4, R19).  The
    gate weight of a chosen pair is the token's softmax probability over the
    experts, p[t, e] (R19).  ``override`` maps an expert to the token set to
    use instead (near ties, as for top-k)."""
    l = np.asarray(logits, np.float64)
    T, E = l.shape
    p = softmax(l)
    tokens = np.empty((E, C), np.int64)
    margin = np.full(E, np.inf)
    for e in range(E):
        order = np.lexsort((np.arange(T), -l[:, e]))   # logit descending, then token
        if 0 < C < T:
            margin[e] = l[order[C - 1], e] - l[order[C], e]
        chosen = order[:C]
        if override is not None and e in override:
            chosen = np.asarray(override[e], np.int64)
        tokens[e] = np.sort(chosen)
    w = p[tokens, np.arange(E)[:, None]]
    return ExpertChoice(C=C, tokens=tokens, w=w, p=p, margin=margin)


# --------------------------------------------------------------------------
# Experts.  [BAIDU] nn.Sequential(Linear(d, d_ff), GELU(), Linear(d_ff, d));
# [SKILLS] §3.1 the same with 4x width; Dropout of the [xdnf] Expert is the
# identity in a forward/eval pass.
# --------------------------------------------------------------------------
def gelu(v: np.ndarray) -> np.ndarray:
    """nn.GELU() default: the exact form 0.5 * v * (1 + erf(v / sqrt(2))) (R8)."""
    v = np.asarray(v, np.float64)
    return 0.5 * v * (1.0 + erf(v / math.sqrt(2.0)))


def silu(v: np.ndarray) -> np.ndarray:
    """nn.SiLU(): v * sigmoid(v), the sigmoid being the logistic function."""
    v = np.asarray(v, np.float64)
    return v * expit(v)


def expert_ffn(xe: np.ndarray, w1: np.ndarray, b1: Optional[np.ndarray],
               w2: np.ndarray, b2: Optional[np.ndarray], act: str = ACT_GELU) -> np.ndarray:
    """y = act(x W1^T + b1) W2^T + b2 with nn.Linear weights W1 [d_ff, d],
    W2 [d, d_ff], in float64; act is GELU or SiLU.

    SwiGLU (R18): W1 is [2 d_ff, d], the gate projection's rows first and the
    up projection's after them (b1 likewise [2 d_ff]); with h = x W1^T + b1
    split into those two halves, y = (SiLU(h_gate) * h_up) W2^T + b2."""
    h = np.asarray(xe, np.float64) @ np.asarray(w1, np.float64).T
    if b1 is not None:
        h = h + np.asarray(b1, np.float64)
    if act == ACT_GELU:
        h = gelu(h)
    elif act == ACT_SILU:
        h = silu(h)
    elif act == ACT_SWIGLU:
        F = h.shape[1] // 2
        h = silu(h[:, :F]) * h[:, F:]
    else:
        raise ValueError(f"unknown activation {act!r}")
    y = h @ np.asarray(w2, np.float64).T
    if b2 is not None:
        y = y + np.asarray(b2, np.float64)
    return y


def expert_ffn_mxfp8(xe: np.ndarray, w1: np.ndarray, b1: Optional[np.ndarray],
                     w2: np.ndarray, b2: Optional[np.ndarray], act: str = ACT_GELU) -> np.ndarray:
    """The expert FFN with MX FP8 operands (R22).

    Both contractions take their two operands MX-quantised along the
    contraction axis: x rows and W1 rows along d for the first, the hidden
    activation's rows and W2 rows along d_ff for the second.  The hidden
    activation act(x W1^T + b1) is formed in float64 from the quantised
    operands, rounded to float32 (the precision in which the kernels hold it
    when they quantise it) and quantised.  Biases are not quantised.  The
    products and sums are float64."""
    from . import mxfp8 as mx
    xq = mx.fake_quant(xe)
    w1q = mx.fake_quant(w1)
    h = xq @ w1q.T
    if b1 is not None:
        h = h + np.asarray(b1, np.float64)
    if act == ACT_GELU:
        h = gelu(h)
    elif act == ACT_SILU:
        h = silu(h)
    elif act == ACT_SWIGLU:
        F = h.shape[1] // 2
        h = silu(h[:, :F]) * h[:, F:]
    else:
        raise ValueError(f"unknown activation {act!r}")
    hq = mx.fake_quant(h.astype(np.float32))
    y = hq @ mx.fake_quant(w2).T
    if b2 is not None:
        y = y + np.asarray(b2, np.float64)
    return y


def _ffn_of(cfg: OracleConfig):
    return expert_ffn_mxfp8 if cfg.experts == "mxfp8" else expert_ffn


# --------------------------------------------------------------------------
# Load-balance statistics.  [BEE] load_balance_loss; [BAIDU] gate step 3;
# [CH7] §7.4 L_balance = N * sum f_i p_i.
# --------------------------------------------------------------------------
def load_balance(cfg: OracleConfig, logits: np.ndarray, p: np.ndarray,
                 counts: np.ndarray):
    """f_i, P_i and aux = alpha * E * sum_i f_i P_i.

    * topk_count: f_i = counts_i / T (the [BAIDU] one-hot of the top-k summed
      over the k and averaged over tokens, so sum f = k; reading R1), counted
      before any capacity drop (R2).
    * argmax: f_i = (tokens whose largest logit is expert i) / T ([BEE]).
    P_i = mean over tokens of the unbiased softmax.
    """
    T = p.shape[0]
    if cfg.aux_f == AUX_TOPK_COUNT:
        f = np.asarray(counts, np.float64) / T
    elif cfg.aux_f == AUX_ARGMAX:
        top1 = np.argmax(np.asarray(logits, np.float64), axis=-1)  # first max
        f = np.bincount(top1, minlength=cfg.E).astype(np.float64) / T
    else:
        raise ValueError(cfg.aux_f)
    P = p.mean(axis=0)
    aux = cfg.aux_alpha * cfg.E * float(np.sum(f * P))
    return f, P, aux


def router_z_loss(logits: np.ndarray) -> float:
    """Router z-loss ([SKILLS] §4.3 ``router_z_loss``): the mean over tokens of
    the squared log-sum-exp of the router logits, in float64 from the float32
    logits (max-subtracted, so the value is the textbook
    log(sum_e exp(l_e))^2 averaged over tokens)."""
    l = np.asarray(logits, np.float64)
    if l.shape[0] == 0:
        return 0.0
    m = l.max(axis=-1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(l - m).sum(axis=-1))
    return float(np.mean(lse * lse))


# --------------------------------------------------------------------------
# The whole layer.
# --------------------------------------------------------------------------
ExpertWeights = Callable[[int], tuple]   # e -> (w1, b1, w2, b2), arrays or None


@dataclass
class ForwardResult:
    logits: np.ndarray
    gate: GateResult
    disp: Dispatch
    C: Optional[int]
    f: np.ndarray
    P: np.ndarray
    aux: float
    rows: np.ndarray                 # token ids whose outputs were computed
    out: np.ndarray                  # [len(rows), d] float64
    extra: dict = field(default_factory=dict)


def moe_forward(cfg: OracleConfig, x: np.ndarray, w_g: np.ndarray,
                experts: ExpertWeights, shared: Optional[ExpertWeights] = None,
                logit_bias: Optional[np.ndarray] = None,
                select_bias: Optional[np.ndarray] = None,
                rows: Optional[Sequence[int]] = None,
                idx_override: Optional[dict] = None) -> ForwardResult:
    """MoE(x_t) = sum over kept j of w[t,j] * E_{idx[t,j]}(x_t)
                 + sum over shared s of S_s(x_t)

    ([CH7] §7.1 formula; [BAIDU] SimpleMoELayer.forward; [SKILLS] §7.1
    ``shared_output + routed_output`` with shared weight one, R12).

    Routing, statistics and dispatch always cover all T tokens (capacity ranks
    depend on every token).  The expert FFNs are evaluated for the tokens in
    ``rows`` only (default: all), one expert at a time, on exactly the rows
    that expert keeps; ``experts(e)`` supplies that expert's weights so a caller
    may fetch them lazily.
    """
    x = np.asarray(x)
    T = x.shape[0]
    assert T == cfg.T
    logits = router_logits(x, w_g, logit_bias)
    if cfg.route == ROUTE_EXPERT_CHOICE:
        return _expert_choice_forward(cfg, x, logits, experts, shared, rows, idx_override)
    g = gate(logits, cfg, select_bias, idx_override)
    C = capacity(cfg)
    disp = dispatch(g.idx, cfg.E, C)
    f, P, aux = load_balance(cfg, logits, g.p, disp.counts)
    z = router_z_loss(logits)

    rows = np.arange(T) if rows is None else np.asarray(rows, np.int64)
    out = np.zeros((len(rows), cfg.d_model), np.float64)
    x64_rows = np.asarray(x[rows], np.float64)

    # assignments (position in rows, slot j) of the requested rows
    a = rows[:, None] * cfg.k + np.arange(cfg.k)[None, :]
    e_of = g.idx.reshape(-1)[a]
    kept = disp.slot_of[a] >= 0
    for e in range(cfg.E):
        ii, jj = np.nonzero((e_of == e) & kept)
        if ii.size == 0:
            continue
        w1, b1, w2, b2 = experts(e)
        y = _ffn_of(cfg)(x64_rows[ii], w1, b1, w2, b2, act=cfg.act)
        wt = g.w[rows[ii], jj][:, None]
        np.add.at(out, ii, wt * y)          # index_add_ of the weighted outputs

    for s in range(cfg.n_shared):
        w1, b1, w2, b2 = shared(s)
        out += _ffn_of(cfg)(x64_rows, w1, b1, w2, b2, act=cfg.act)

    return ForwardResult(logits=logits, gate=g, disp=disp, C=C, f=f, P=P,
                         aux=aux, rows=rows, out=out, extra={"z_loss": z})


def _expert_choice_forward(cfg, x, logits, experts, shared, rows, override):
    """The layer under Expert Choice routing:
    MoE(x_t) = sum over experts e that chose t of p[t, e] * E_e(x_t)
               + sum over shared s of S_s(x_t).
    Statistics: every expert processes exactly C tokens, so with topk_count
    f_e = C / T; P and aux as for top-k routing.  ``disp`` lists the experts'
    rows in order (offsets e * C); its per-assignment fields are empty."""
    T, E = logits.shape
    C = expert_choice_capacity(cfg)
    ec = expert_choice(logits, C, override)
    counts = np.full(E, C, np.int64)
    f, P, aux = load_balance(cfg, logits, ec.p, counts)
    z = router_z_loss(logits)
    empty = np.zeros(0, np.int64)
    disp = Dispatch(counts=counts, kept=counts.copy(),
                    offsets=np.arange(E + 1, dtype=np.int64) * C,
                    perm_token=ec.tokens.reshape(-1).copy(), slot_of=empty, rank=empty)

    rows = np.arange(T) if rows is None else np.asarray(rows, np.int64)
    out = np.zeros((len(rows), cfg.d_model), np.float64)
    x64_rows = np.asarray(x[rows], np.float64)
    pos_of = {int(t): i for i, t in enumerate(rows)}
    for e in range(E):
        pick = [(pos_of[int(t)], j) for j, t in enumerate(ec.tokens[e]) if int(t) in pos_of]
        if not pick:
            continue
        ii = np.array([a for a, _ in pick], np.int64)
        jj = np.array([b for _, b in pick], np.int64)
        w1, b1, w2, b2 = experts(e)
        y = _ffn_of(cfg)(x64_rows[ii], w1, b1, w2, b2, act=cfg.act)
        np.add.at(out, ii, ec.w[e, jj][:, None] * y)
    for s in range(cfg.n_shared):
        w1, b1, w2, b2 = shared(s)
        out += _ffn_of(cfg)(x64_rows, w1, b1, w2, b2, act=cfg.act)
    return ForwardResult(logits=logits, gate=None, disp=disp, C=C, f=f, P=P, aux=aux,
                         rows=rows, out=out, extra={"z_loss": z, "ec": ec})
