"""Comparison of a device run of the MoE layer with the oracle.

TEST INFRASTRUCTURE ONLY (used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``).  It imports nothing from the product
package: device results arrive as torch tensors or numpy arrays.

Acceptance rules:
* expert indices, per-expert counts, kept counts, offsets, the permutation and
  the dropped set are bit-exact, except for tokens whose neighbouring
  selection scores (among the k+1 best) are closer than NEAR_TIE; those are
  reported, and the oracle is re-run with the device's choice for them so
  that everything downstream is still compared exactly;
* f is exact (a ratio of integers, compared after rounding the oracle's value
  to float32), P and aux within 1e-5 relative, gate weights within 1e-5;
* layer output: relative L2 <= 1e-2 and max-abs <= 5e-2 x RMS(reference) for
  bf16 layers; relative L2 <= 1e-4 for fp32 layers.  Reference rows that are
  exactly zero (every assignment of the token dropped) must be exactly zero,
  and RMS is taken over the other rows.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

from . import moe_oracle as om

NEAR_TIE = 1e-5
TOL_BF16_REL_L2 = 1e-2
TOL_BF16_MAX_ABS_RMS = 5e-2
TOL_F32_REL_L2 = 1e-4
TOL_P_REL = 1e-5
TOL_AUX_REL = 1e-5
TOL_W_ABS = 1e-5
# router z-loss: each token's log-sum-exp is 1-Lipschitz in the logits, which
# agree to about 1e-6 relative (fp32 dot products); squaring doubles that and
# the fp32 mean over T tokens in blocked order adds a few 1e-7 more.
TOL_Z_REL = 1e-4


def oracle_config(cfg: dict) -> om.OracleConfig:
    """The oracle's view of a workload dict.  The capacity factor is rounded to
    float32 first: that is the value the library receives."""
    return om.OracleConfig(
        T=int(cfg["T"]), d_model=int(cfg["d_model"]), d_ff=int(cfg["d_ff"]), E=int(cfg["E"]),
        k=int(cfg["k"]), n_shared=int(cfg.get("n_shared", 0)),
        capacity_factor=float(np.float32(cfg.get("capacity_factor", 0.0))),
        min_capacity=int(cfg.get("min_capacity", 0)), route=cfg["route"],
        renorm=bool(cfg.get("renorm", 1)),
        aux_alpha=float(np.float32(cfg.get("aux_alpha", 0.01))),
        aux_f=cfg.get("aux_f", om.AUX_TOPK_COUNT), act=cfg.get("act", om.ACT_GELU),
        experts=cfg.get("experts", "dense"))


def np64(t) -> Optional[np.ndarray]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def np32(t) -> Optional[np.ndarray]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float32)
    return t.detach().to("cpu", torch.float32).numpy()


class LazyExperts:
    """expert e -> (w1, b1, w2, b2) in float64, copied from the (device)
    tensors one expert at a time, so full-size layers never hold every
    expert in float64 on the host at once."""

    def __init__(self, w1, b1, w2, b2):
        self.w1, self.b1, self.w2, self.b2 = w1, b1, w2, b2

    def __call__(self, e: int):
        return (np64(self.w1[e]), None if self.b1 is None else np64(self.b1[e]),
                np64(self.w2[e]), None if self.b2 is None else np64(self.b2[e]))


def run_oracle(cfg: dict, inputs: dict, rows: Optional[Sequence[int]] = None,
               idx_override: Optional[dict] = None) -> om.ForwardResult:
    ocfg = oracle_config(cfg)
    experts = LazyExperts(inputs["w1"], inputs.get("b1"), inputs["w2"], inputs.get("b2"))
    shared = None
    if ocfg.n_shared:
        shared = LazyExperts(inputs["ws1"], inputs.get("wsb1"), inputs["ws2"], inputs.get("wsb2"))
    return om.moe_forward(ocfg, np64(inputs["x"]), np64(inputs["w_g"]), experts, shared,
                          logit_bias=np32(inputs.get("logit_bias")),
                          select_bias=np64(inputs.get("select_bias")),
                          rows=rows, idx_override=idx_override)


@dataclass
class Report:
    near_tie: list = field(default_factory=list)       # tokens within NEAR_TIE
    overridden: list = field(default_factory=list)     # near-tie tokens whose choice differs
    rel_l2: float = 0.0
    max_abs_over_rms: float = 0.0
    checked_rows: int = 0
    notes: list = field(default_factory=list)

    def summary(self) -> str:
        return (f"rows={self.checked_rows} rel_l2={self.rel_l2:.3e} "
                f"maxabs/rms={self.max_abs_over_rms:.3e} near_tie={len(self.near_tie)} "
                f"overridden={len(self.overridden)}")


def _near_tie_and_override(ref: om.ForwardResult, gpu_idx: np.ndarray):
    """Near-tie tokens, and the device's choice for those among them where it
    differs from the oracle's.  Such a choice must still be a valid top-k up to
    the margin: k distinct experts in [0, E), each scoring at least the k-th
    best score minus NEAR_TIE, listed in descending score up to NEAR_TIE."""
    nt = np.nonzero(ref.gate.margin < NEAR_TIE)[0]
    override = {}
    E = ref.gate.p.shape[1]
    for t in nt:
        if np.array_equal(gpu_idx[t], ref.gate.idx[t]):
            continue
        g = np.asarray(gpu_idx[t]).astype(np.int64)
        k = g.size
        assert np.all((g >= 0) & (g < E)) and len(set(g.tolist())) == k, \
            f"token {t}: device experts {g.tolist()} are not k distinct experts"
        sc = ref.gate.score[t]
        kth = np.sort(sc)[::-1][k - 1]
        assert sc[g].min() >= kth - NEAR_TIE, \
            f"token {t}: device experts {g.tolist()} are not a top-{k} set (scores {sc[g]})"
        assert np.all(sc[g][:-1] >= sc[g][1:] - NEAR_TIE), \
            f"token {t}: device experts {g.tolist()} are not in descending score order"
        override[int(t)] = g
    return [int(t) for t in nt], override


def compare_routing(cfg: dict, ref: om.ForwardResult, gpu: dict, rep: Report) -> None:
    """idx / w / counts / f / P / aux / z_loss (the dict holds numpy arrays)."""
    idx = np.asarray(gpu["topk_idx"]).astype(np.int64)
    T = idx.shape[0]
    ok = np.ones(T, bool)
    ok[list(rep.overridden)] = False
    bad = np.nonzero(np.any(idx != ref.gate.idx, axis=1) & ok)[0]
    assert bad.size == 0, (f"expert indices differ on {bad.size} tokens outside the near-tie "
                           f"set, e.g. t={bad[:5].tolist()}: gpu={idx[bad[:3]].tolist()} "
                           f"oracle={ref.gate.idx[bad[:3]].tolist()} "
                           f"margin={ref.gate.margin[bad[:3]].tolist()}")
    if "topk_w" in gpu:
        dw = np.abs(np.asarray(gpu["topk_w"], np.float64) - ref.gate.w)
        assert dw.max() <= TOL_W_ABS, f"gate weights differ by {dw.max():.3e}"
    if "counts" in gpu:
        assert np.array_equal(np.asarray(gpu["counts"]).astype(np.int64), ref.disp.counts), \
            "per-expert counts differ"
    if "f" in gpu:
        f_ref = ref.f.astype(np.float32)
        f_gpu = np.asarray(gpu["f"], np.float32)
        if ref.gate is not None and oracle_config(cfg).aux_f == om.AUX_ARGMAX and rep.near_tie:
            slack = len(rep.near_tie) / T
            assert np.max(np.abs(f_gpu - f_ref)) <= slack + 1e-7, "f differs"
        else:
            assert np.array_equal(f_gpu, f_ref), \
                f"f differs: max {np.max(np.abs(f_gpu - f_ref))}"
    if "P" in gpu:
        P = np.asarray(gpu["P"], np.float64)
        err = np.abs(P - ref.P) / np.maximum(np.abs(ref.P), 1e-30)
        assert err.max() <= TOL_P_REL, f"P relative error {err.max():.3e}"
    if "aux" in gpu:
        a = float(np.asarray(gpu["aux"]).reshape(-1)[0])
        slack = 0.0
        if oracle_config(cfg).aux_f == om.AUX_ARGMAX and rep.near_tie:
            slack = cfg["aux_alpha"] * cfg["E"] * len(rep.near_tie) / T
        assert abs(a - ref.aux) <= TOL_AUX_REL * abs(ref.aux) + slack + 1e-12, \
            f"aux {a} vs {ref.aux}"
    if gpu.get("z_loss") is not None and "z_loss" in ref.extra:
        z = float(np.asarray(gpu["z_loss"]).reshape(-1)[0])
        zr = float(ref.extra["z_loss"])
        assert abs(z - zr) <= TOL_Z_REL * abs(zr) + 1e-12, f"z_loss {z} vs {zr}"


def compare_dispatch(ref: om.ForwardResult, gpu: dict) -> None:
    """kept / offsets / perm_token / slot_of bit-exact; x_perm rows = x[perm_token]."""
    d = ref.disp
    if "kept" in gpu:
        assert np.array_equal(np.asarray(gpu["kept"]).astype(np.int64), d.kept), "kept differs"
    if "offsets" in gpu:
        assert np.array_equal(np.asarray(gpu["offsets"]).astype(np.int64), d.offsets), \
            "offsets differ"
    n = int(d.offsets[-1])
    if "perm_token" in gpu:
        assert np.array_equal(np.asarray(gpu["perm_token"])[:n].astype(np.int64),
                              d.perm_token), "perm_token differs"
    if "slot_of" in gpu:
        assert np.array_equal(np.asarray(gpu["slot_of"]).astype(np.int64), d.slot_of), \
            "slot_of (kept rows / dropped set) differs"


def compare_output(cfg: dict, ref: om.ForwardResult, out_gpu: np.ndarray, rep: Report) -> None:
    """Rows whose reference is exactly zero (every assignment dropped, no
    shared expert) must be exactly zero; the other rows meet the tolerance,
    with RMS taken over them (the same as the plain rule when nothing drops)."""
    o = np.asarray(out_gpu, np.float64)[ref.rows]
    r = ref.out
    zero = ~np.any(r != 0.0, axis=1) if r.size else np.zeros(0, bool)
    if zero.any():
        assert np.all(o[zero] == 0.0), "rows with every assignment dropped must be 0"
    o, r = o[~zero], r[~zero]
    rep.checked_rows = len(ref.rows)
    if not r.size:
        return
    diff = o - r
    rms = float(np.sqrt(np.mean(r * r)))
    rel = float(np.linalg.norm(diff) / np.linalg.norm(r))
    mx = float(np.max(np.abs(diff)) / rms)
    rep.rel_l2, rep.max_abs_over_rms = rel, mx
    if cfg["dtype"] == "f32":
        assert rel <= TOL_F32_REL_L2, f"fp32 rel-L2 {rel:.3e} > {TOL_F32_REL_L2}"
    else:
        assert rel <= TOL_BF16_REL_L2, f"bf16 rel-L2 {rel:.3e} > {TOL_BF16_REL_L2}"
        assert mx <= TOL_BF16_MAX_ABS_RMS, f"bf16 max-abs/RMS {mx:.3e} > {TOL_BF16_MAX_ABS_RMS}"


def compare_stats(cfg: dict, ref: om.ForwardResult, gpu: dict) -> None:
    """f exact; P, aux and z_loss within their tolerances (no near-tie slack)."""
    if "f" in gpu:
        f_gpu = np.asarray(gpu["f"], np.float32)
        assert np.array_equal(f_gpu, ref.f.astype(np.float32)), "f differs"
    if "P" in gpu:
        P = np.asarray(gpu["P"], np.float64)
        err = np.abs(P - ref.P) / np.maximum(np.abs(ref.P), 1e-30)
        assert err.max() <= TOL_P_REL, f"P relative error {err.max():.3e}"
    if "aux" in gpu:
        a = float(np.asarray(gpu["aux"]).reshape(-1)[0])
        assert abs(a - ref.aux) <= TOL_AUX_REL * abs(ref.aux) + 1e-12, f"aux {a} vs {ref.aux}"
    if gpu.get("z_loss") is not None:
        z = float(np.asarray(gpu["z_loss"]).reshape(-1)[0])
        zr = float(ref.extra["z_loss"])
        assert abs(z - zr) <= TOL_Z_REL * abs(zr) + 1e-12, f"z_loss {z} vs {zr}"


def check_layer_expert_choice(cfg: dict, inputs: dict, gpu: dict,
                              rows: Optional[Sequence[int]] = None) -> Report:
    """Expert Choice: each expert's taken tokens bit-exact, except experts
    whose C-th and (C+1)-th largest logits are closer than NEAR_TIE.  For
    those the device's set must still be a top-C up to that margin, and the
    oracle is re-run with it.  ``gpu`` holds topk_idx / topk_w as [E, C]
    token lists and weights, counts, f, P, aux, z_loss and out."""
    rep = Report()
    ref = run_oracle(cfg, inputs, rows=rows)
    ec = ref.extra["ec"]
    C, E = ec.C, cfg["E"]
    tok = np.asarray(gpu["topk_idx"]).astype(np.int64).reshape(E, C)
    rep.near_tie = [int(e) for e in np.nonzero(ec.margin < NEAR_TIE)[0]]
    override = {}
    for e in range(E):
        if np.array_equal(tok[e], ec.tokens[e]):
            continue
        assert ec.margin[e] < NEAR_TIE, (
            f"expert {e} took other tokens (margin {ec.margin[e]:.3e}): "
            f"gpu-only {sorted(set(tok[e]) - set(ec.tokens[e]))[:5]} "
            f"oracle-only {sorted(set(ec.tokens[e]) - set(tok[e]))[:5]}")
        col = ref.logits[:, e]
        kth = np.sort(col)[::-1][C - 1]
        assert len(set(tok[e].tolist())) == C and np.all(np.diff(tok[e]) > 0)
        assert col[tok[e]].min() >= kth - NEAR_TIE, f"expert {e}: not a top-C set"
        override[e] = tok[e]
    if override:
        rep.overridden = sorted(override)
        ref = run_oracle(cfg, inputs, rows=rows, idx_override=override)
        ec = ref.extra["ec"]
    if "topk_w" in gpu:
        dw = np.abs(np.asarray(gpu["topk_w"], np.float64).reshape(E, C) - ec.w)
        assert dw.size == 0 or dw.max() <= TOL_W_ABS, f"gate weights differ by {dw.max():.3e}"
    if "counts" in gpu:
        assert np.all(np.asarray(gpu["counts"]) == C), "counts must all be C"
    compare_stats(cfg, ref, gpu)
    if "out" in gpu:
        compare_output(cfg, ref, gpu["out"], rep)
    return rep


def check_layer(cfg: dict, inputs: dict, gpu: dict, rows: Optional[Sequence[int]] = None
                ) -> Report:
    """Full acceptance check of one device run against the oracle.

    ``gpu`` maps output names to numpy arrays: topk_idx, topk_w, counts, f, P,
    aux, out (and optionally kept, offsets, perm_token, slot_of)."""
    if cfg.get("route") == om.ROUTE_EXPERT_CHOICE:
        return check_layer_expert_choice(cfg, inputs, gpu, rows)
    rep = Report()
    ref = run_oracle(cfg, inputs, rows=rows)
    rep.near_tie, override = _near_tie_and_override(ref, np.asarray(gpu["topk_idx"]))
    if override:
        rep.overridden = sorted(override)
        ref = run_oracle(cfg, inputs, rows=rows, idx_override=override)
    compare_routing(cfg, ref, gpu, rep)
    compare_dispatch(ref, gpu)
    if "out" in gpu:
        compare_output(cfg, ref, gpu["out"], rep)
    return rep
