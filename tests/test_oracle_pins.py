"""Pins for the CPU oracle: facts the pages and the mathematics fix, checked
independently of the oracle's own code paths.

Each ``check_*`` function is a pin; the ``test_*`` functions run them, and the
``test_plant_*`` functions plant a plausible mistake in the oracle (on the CPU)
and show that at least one pin fails.
"""

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.moe_oracle as om
from oracle.moe_oracle import OracleConfig

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")
LN3 = math.log(3.0)


def _cfg(**kw):
    base = dict(T=16, d_model=8, d_ff=12, E=4, k=2)
    base.update(kw)
    return OracleConfig(**base)


def _rand_layer(rng, T, d, F, E, S=0, bias=True):
    x = rng.standard_normal((T, d))
    w_g = rng.standard_normal((d, E)) / math.sqrt(d)
    ex = [(rng.standard_normal((F, d)) / math.sqrt(d),
           rng.standard_normal(F) * 0.1 if bias else None,
           rng.standard_normal((d, F)) / math.sqrt(F),
           rng.standard_normal(d) * 0.1 if bias else None) for _ in range(E)]
    sh = [(rng.standard_normal((F, d)) / math.sqrt(d), None,
           rng.standard_normal((d, F)) / math.sqrt(F), None) for _ in range(S)]
    return x, w_g, ex, sh


def _torch_ffn(x, w1, b1, w2, b2):
    """Textbook two-layer MLP through torch's own Linear and exact GELU."""
    t = lambda a: None if a is None else torch.as_tensor(np.asarray(a), dtype=torch.float64)
    h = torch.nn.functional.linear(t(x), t(w1), t(b1))
    h = torch.nn.functional.gelu(h, approximate="none")
    return torch.nn.functional.linear(h, t(w2), t(b2)).numpy()


# ---------------------------------------------------------------- golden
def check_golden_pages_values():
    g = json.load(open(GOLDEN))
    for item in g["expert_combinations"]:
        assert math.comb(item["E"], item["k"]) == item["count"], item
        if item["count"] < 10 ** 6:
            # the brute-force selection enumerates exactly these subsets
            assert len(_subsets(item["E"], item["k"])) == item["count"]
    for item in g["activated_fraction"]:
        assert abs(item["k"] / item["E"] - item["fraction"]) <= item["abs_tol"] + 1e-15
    for item in g["experts_per_token_with_shared"]:
        assert item["n_shared"] + item["k"] == item["total"]
    for item in g["capacity"]:
        cfg = OracleConfig(T=item["T"], d_model=1, d_ff=1, E=item["E"], k=1,
                           capacity_factor=item["capacity_factor"])
        assert om.capacity(cfg) == item["C"], item


def test_golden_pages_values():
    check_golden_pages_values()


# ---------------------------------------------------------------- selection
def _subsets(E, k):
    return list(itertools.combinations(range(E), k))


def _brute_select(score_row, k):
    """Enumerate every k-subset; keep the largest score sum, breaking equal
    sums by the lexicographically smallest index tuple."""
    best, best_sum = None, None
    for sub in _subsets(len(score_row), k):     # lexicographic order
        # exact rational sums: float rounding must not break equal sums
        s = sum(Fraction(float(score_row[i])) for i in sub)
        if best_sum is None:
            best, best_sum = sub, s
        if s > best_sum:
            best, best_sum = sub, s
    return best


def check_selection_bruteforce(seed=0):
    rng = np.random.default_rng(seed)
    for E, k in [(4, 1), (4, 2), (5, 3), (8, 2), (8, 3)]:
        for trial in range(6):
            # scores on a coarse grid so that ties occur often
            l = rng.integers(-3, 4, size=(12, E)).astype(np.float32)
            for route in (om.ROUTE_SOFTMAX_TOPK, om.ROUTE_TOPK_SOFTMAX, om.ROUTE_BIASED_SOFTMAX):
                sb = rng.integers(0, 3, size=E) * 0.25 if route == om.ROUTE_BIASED_SOFTMAX else None
                cfg = _cfg(T=12, E=E, k=k, route=route)
                g = om.gate(l, cfg, select_bias=sb)
                p = np.exp(l.astype(np.float64))
                p /= p.sum(1, keepdims=True)
                if route == om.ROUTE_SOFTMAX_TOPK:
                    score = p
                elif route == om.ROUTE_TOPK_SOFTMAX:
                    score = l.astype(np.float64)
                else:
                    score = p + sb
                for t in range(12):
                    want = _brute_select(list(score[t]), k)
                    got = tuple(sorted(int(i) for i in g.idx[t]))
                    assert got == want, (route, E, k, t, score[t], got, want)
                    # order: descending score, ties by ascending index
                    row = [(-score[t][i], int(i)) for i in g.idx[t]]
                    assert row == sorted(row), (route, t, row)


def test_selection_bruteforce():
    check_selection_bruteforce()


def check_hand_gate_examples():
    # logits ln[4,2,1,1] -> p = [.5,.25,.125,.125]; top-2 = {0,1}
    l = np.log(np.array([[4.0, 2.0, 1.0, 1.0]], np.float32)).astype(np.float32)
    g = om.gate(l, _cfg(T=1, E=4, k=2, route=om.ROUTE_SOFTMAX_TOPK))
    assert list(g.idx[0]) == [0, 1]
    np.testing.assert_allclose(g.w[0], [2 / 3, 1 / 3], rtol=1e-6)
    np.testing.assert_allclose(g.p[0], [0.5, 0.25, 0.125, 0.125], rtol=1e-6)
    # without renormalisation the weights are the probabilities themselves
    g = om.gate(l, _cfg(T=1, E=4, k=2, route=om.ROUTE_SOFTMAX_TOPK, renorm=False))
    np.testing.assert_allclose(g.w[0], [0.5, 0.25], rtol=1e-6)
    # top-k on logits, softmax over the two: exp(ln4)/(4+2) = 2/3
    g = om.gate(l, _cfg(T=1, E=4, k=2, route=om.ROUTE_TOPK_SOFTMAX))
    assert list(g.idx[0]) == [0, 1]
    np.testing.assert_allclose(g.w[0], [2 / 3, 1 / 3], rtol=1e-6)
    # selection bias 0.2 on expert 2: scores [.5,.25,.325,.125] -> {0,2};
    # weights from the unbiased p: .5/.625, .125/.625
    g = om.gate(l, _cfg(T=1, E=4, k=2, route=om.ROUTE_BIASED_SOFTMAX),
                select_bias=np.array([0.0, 0.0, 0.2, 0.0]))
    assert list(g.idx[0]) == [0, 2]
    np.testing.assert_allclose(g.w[0], [0.8, 0.2], rtol=1e-6)
    # all-equal logits: lowest indices win, equal weights
    g = om.gate(np.zeros((1, 4), np.float32), _cfg(T=1, E=4, k=2))
    assert list(g.idx[0]) == [0, 1]
    np.testing.assert_allclose(g.w[0], [0.5, 0.5], rtol=0, atol=0)


def test_hand_gate_examples():
    check_hand_gate_examples()


def check_softmax_topk_equals_topk_softmax(seed=1):
    """softmax(l)_i / sum_S softmax(l)_j = exp(l_i) / sum_S exp(l_j): with
    renormalisation, both gating forms give the same experts and weights."""
    rng = np.random.default_rng(seed)
    for E, k in [(8, 2), (64, 1), (16, 4), (256, 8)]:
        l = (rng.standard_normal((64, E)) * 2).astype(np.float32)
        a = om.gate(l, _cfg(T=64, E=E, k=k, route=om.ROUTE_SOFTMAX_TOPK, renorm=True))
        b = om.gate(l, _cfg(T=64, E=E, k=k, route=om.ROUTE_TOPK_SOFTMAX))
        ok = a.margin > 1e-9
        assert np.array_equal(a.idx[ok], b.idx[ok])
        np.testing.assert_allclose(a.w[ok], b.w[ok], rtol=1e-12, atol=1e-15)


def test_softmax_topk_equals_topk_softmax():
    check_softmax_topk_equals_topk_softmax()


def check_weights_sum_to_one(seed=2):
    rng = np.random.default_rng(seed)
    for route in (om.ROUTE_SOFTMAX_TOPK, om.ROUTE_TOPK_SOFTMAX, om.ROUTE_BIASED_SOFTMAX):
        for E, k in [(8, 2), (8, 1), (32, 5)]:
            l = rng.standard_normal((50, E)).astype(np.float32)
            g = om.gate(l, _cfg(T=50, E=E, k=k, route=route),
                        select_bias=rng.standard_normal(E) * 0.01)
            np.testing.assert_allclose(g.w.sum(1), 1.0, rtol=0, atol=1e-12)
            if k == 1:
                assert np.all(g.w == 1.0)
            assert np.all(g.w > 0)


def test_weights_sum_to_one():
    check_weights_sum_to_one()


def check_softmax_basic():
    l = np.array([[1000.0, 1000.0, -1000.0], [0.0, LN3, 0.0]], np.float32)
    p = om.softmax(l)
    assert np.all(np.isfinite(p))
    np.testing.assert_allclose(p[0], [0.5, 0.5, 0.0], atol=1e-300)
    np.testing.assert_allclose(p[1], [0.2, 0.6, 0.2], rtol=1e-6)


def test_softmax_basic():
    check_softmax_basic()


def check_router_logits(seed=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((20, 24)).astype(np.float32)
    w = rng.standard_normal((24, 5)).astype(np.float32)
    l = om.router_logits(x, w)
    assert l.dtype == np.float32 and l.shape == (20, 5)
    ref = (torch.from_numpy(x).double() @ torch.from_numpy(w).double()).float().numpy()
    assert np.array_equal(l, ref)
    b = np.arange(5, dtype=np.float32)
    assert np.array_equal(om.router_logits(x, w, b), (ref + b).astype(np.float32))


def test_router_logits():
    check_router_logits()


# ---------------------------------------------------------------- experts
def check_gelu_closed_form():
    # GELU(x) = x * Phi(x); Phi(1) and Phi(-1) of the standard normal CDF
    v = om.gelu(np.array([0.0, 1.0, -1.0, 8.0, -8.0]))
    np.testing.assert_allclose(v[:3], [0.0, 0.8413447460685429, -0.15865525393145707],
                               rtol=1e-15, atol=1e-16)
    np.testing.assert_allclose(v[3], 8.0, rtol=1e-14)
    assert abs(v[4]) < 1e-13


def test_gelu_closed_form():
    check_gelu_closed_form()


def check_silu_closed_form():
    """SiLU(v) = v * sigmoid(v): sigmoid(log 3) = 3/4 exactly, so SiLU(log 3)
    = 0.75 log 3; SiLU(0) = 0; SiLU(v) - SiLU(-v) = v for every v (sigmoid(v)
    + sigmoid(-v) = 1); SiLU(40) = 40 to double precision, SiLU(-40) ~ -40 e^-40."""
    v = om.silu(np.array([LN3, 0.0, 40.0, -40.0]))
    assert abs(v[0] - 0.75 * LN3) < 1e-15
    assert v[1] == 0.0
    assert abs(v[2] - 40.0) < 1e-12
    assert abs(v[3] + 40.0 * math.exp(-40.0)) < 1e-25
    r = np.random.default_rng(11).standard_normal(50) * 4
    np.testing.assert_allclose(om.silu(r) - om.silu(-r), r, rtol=0, atol=1e-14)


def test_silu_closed_form():
    check_silu_closed_form()


def check_glu_experts(seed=12):
    """Hand values of the SiLU and SwiGLU experts, and the special case of
    SwiGLU that reduces to the SiLU expert.
    d = d_ff = 1, x = 1: a SiLU expert with W1 = log 3, W2 = 1 gives 0.75 log 3;
    a SwiGLU expert with gate row log 3, up row 2 gives SiLU(log 3) * 2
    = 1.5 log 3 (the halves the other way round would give 2 sigmoid(2) log 3).
    With the up rows zero and the up bias one, SwiGLU equals the SiLU expert of
    the gate rows."""
    one = np.ones((1, 1))
    y = om.expert_ffn(one, np.array([[LN3]]), None, one, None, act=om.ACT_SILU)
    assert abs(y[0, 0] - 0.75 * LN3) < 1e-15
    y = om.expert_ffn(one, np.array([[LN3], [2.0]]), None, one, None, act=om.ACT_SWIGLU)
    assert abs(y[0, 0] - 1.5 * LN3) < 1e-15, y
    rng = np.random.default_rng(seed)
    T, d, F = 9, 5, 7
    x = rng.standard_normal((T, d))
    wg_rows, bg = rng.standard_normal((F, d)), rng.standard_normal(F)
    w2, b2 = rng.standard_normal((d, F)), rng.standard_normal(d)
    w1 = np.concatenate([wg_rows, np.zeros((F, d))])
    b1 = np.concatenate([bg, np.ones(F)])
    np.testing.assert_allclose(om.expert_ffn(x, w1, b1, w2, b2, act=om.ACT_SWIGLU),
                               om.expert_ffn(x, wg_rows, bg, w2, b2, act=om.ACT_SILU),
                               rtol=1e-14, atol=1e-14)
    # through torch's own SiLU for the plain SiLU expert
    t = lambda a: torch.as_tensor(a, dtype=torch.float64)
    want = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(t(x), t(wg_rows), t(bg))),
        t(w2), t(b2)).numpy()
    np.testing.assert_allclose(om.expert_ffn(x, wg_rows, bg, w2, b2, act=om.ACT_SILU), want,
                               rtol=1e-13, atol=1e-13)
    # the layer applies the configured activation to routed and shared experts
    E = 3
    w1s = [rng.standard_normal((2 * F, d)) for _ in range(E)]
    ex = {e: (w1s[e], None, w2, None) for e in range(E)}
    cfg = om.OracleConfig(T=T, d_model=d, d_ff=F, E=E, k=1, n_shared=1, act=om.ACT_SWIGLU)
    r = om.moe_forward(cfg, x, rng.standard_normal((d, E)), lambda e: ex[e],
                       shared=lambda s: ex[0])
    for t_ in range(T):
        e = int(r.gate.idx[t_, 0])
        h1 = x[t_] @ w1s[e].T
        h0 = x[t_] @ w1s[0].T
        routed = (h1[:F] / (1 + np.exp(-h1[:F])) * h1[F:]) @ w2.T
        shared = (h0[:F] / (1 + np.exp(-h0[:F])) * h0[F:]) @ w2.T
        np.testing.assert_allclose(r.out[t_], r.gate.w[t_, 0] * routed + shared,
                                   rtol=1e-12, atol=1e-12)


def test_glu_experts():
    check_glu_experts()


def check_dense_reductions(seed=4):
    rng = np.random.default_rng(seed)
    T, d, F = 10, 6, 10
    # E = 1, k = 1: the layer is one dense FFN (weight 1 after renormalising)
    x, w_g, ex, _ = _rand_layer(rng, T, d, F, 1)
    r = om.moe_forward(_cfg(T=T, d_model=d, d_ff=F, E=1, k=1), x, w_g, lambda e: ex[e])
    np.testing.assert_allclose(r.out, _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)
    # identical experts + renormalised top-k: FFN(x) whatever the router says
    E = 6
    x, w_g, ex, _ = _rand_layer(rng, T, d, F, E)
    for route in (om.ROUTE_SOFTMAX_TOPK, om.ROUTE_TOPK_SOFTMAX, om.ROUTE_BIASED_SOFTMAX):
        r = om.moe_forward(_cfg(T=T, d_model=d, d_ff=F, E=E, k=3, route=route),
                           x, w_g, lambda e: ex[0],
                           select_bias=rng.standard_normal(E) * 0.01)
        np.testing.assert_allclose(r.out, _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)
    # one shared expert equal to the routed ones: 2 * FFN(x)
    r = om.moe_forward(_cfg(T=T, d_model=d, d_ff=F, E=E, k=2, n_shared=1,
                            route=om.ROUTE_BIASED_SOFTMAX),
                       x, w_g, lambda e: ex[0], shared=lambda s: ex[0],
                       select_bias=rng.standard_normal(E) * 0.01)
    np.testing.assert_allclose(r.out, 2 * _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)


def test_dense_reductions():
    check_dense_reductions()


# ---------------------------------------------------------------- aux loss
def check_aux_uniform_router():
    """W_g = 0 makes every p = 1/E, so aux = alpha * E * sum f_i / E = k * alpha
    for any f (sum f = k)."""
    rng = np.random.default_rng(5)
    for E, k, route in [(8, 2, om.ROUTE_SOFTMAX_TOPK), (64, 1, om.ROUTE_SOFTMAX_TOPK),
                        (16, 4, om.ROUTE_TOPK_SOFTMAX), (256, 8, om.ROUTE_BIASED_SOFTMAX)]:
        T, d = 32, 8
        x = rng.standard_normal((T, d))
        cfg = _cfg(T=T, d_model=d, d_ff=4, E=E, k=k, route=route, aux_alpha=0.01)
        l = om.router_logits(x, np.zeros((d, E)))
        g = om.gate(l, cfg, select_bias=rng.standard_normal(E) * 0.01)
        disp = om.dispatch(g.idx, E, None)
        f, P, aux = om.load_balance(cfg, l, g.p, disp.counts)
        np.testing.assert_allclose(P, 1.0 / E, rtol=1e-15)
        assert abs(f.sum() - k) < 1e-12
        assert abs(aux - k * 0.01) < 1e-15


def test_aux_uniform_router():
    check_aux_uniform_router()


def check_aux_hand_example():
    """T=4, E=2, k=1, W_g = I: logits [0,0], [ln3,0], [0,ln3], [0,-ln3].
    p = [.5,.5], [.75,.25], [.25,.75], [.75,.25]; argmax (lowest index on the
    tie) = 0,0,1,0 -> f = [3/4, 1/4]; P = [2.25/4, 1.75/4];
    aux = 0.01 * 2 * (0.75*0.5625 + 0.25*0.4375) = 0.010625."""
    x = np.array([[0, 0], [LN3, 0], [0, LN3], [0, -LN3]], np.float64)
    for aux_f in (om.AUX_ARGMAX, om.AUX_TOPK_COUNT):
        cfg = OracleConfig(T=4, d_model=2, d_ff=1, E=2, k=1, aux_f=aux_f, aux_alpha=0.01)
        l = om.router_logits(x, np.eye(2))
        g = om.gate(l, cfg)
        assert list(g.idx[:, 0]) == [0, 0, 1, 0]
        disp = om.dispatch(g.idx, 2, None)
        f, P, aux = om.load_balance(cfg, l, g.p, disp.counts)
        np.testing.assert_allclose(f, [0.75, 0.25], rtol=0, atol=0)
        np.testing.assert_allclose(P, [0.5625, 0.4375], rtol=1e-7)
        assert abs(aux - 0.010625) < 1e-8


def test_aux_hand_example():
    check_aux_hand_example()


def check_aux_nonnegative_and_argmax(seed=6):
    rng = np.random.default_rng(seed)
    T, d, E = 200, 16, 8
    x = rng.standard_normal((T, d))
    w = rng.standard_normal((d, E))
    l = om.router_logits(x, w)
    a = OracleConfig(T=T, d_model=d, d_ff=4, E=E, k=1, aux_f=om.AUX_ARGMAX)
    b = OracleConfig(T=T, d_model=d, d_ff=4, E=E, k=1, aux_f=om.AUX_TOPK_COUNT)
    g = om.gate(l, a)
    disp = om.dispatch(g.idx, E, None)
    fa, Pa, auxa = om.load_balance(a, l, g.p, disp.counts)
    fb, Pb, auxb = om.load_balance(b, l, g.p, disp.counts)
    # top-1 of the softmax is the argmax of the logits: both f forms agree
    assert np.array_equal(fa, fb) and auxa == auxb and auxa >= 0


def test_aux_nonnegative_and_argmax():
    check_aux_nonnegative_and_argmax()


# ---------------------------------------------------------------- dispatch
def check_capacity_hand_example():
    """T=8, E=2, k=1, CF=0.5 -> C = floor(0.5*8/2) = 2.  idx = 1,0,1,1,0,1,0,0:
    expert 0 sees tokens 1,4,6,7 and keeps 1,4; expert 1 sees 0,2,3,5 and
    keeps 0,2."""
    cfg = OracleConfig(T=8, d_model=1, d_ff=1, E=2, k=1, capacity_factor=0.5)
    C = om.capacity(cfg)
    assert C == 2
    idx = np.array([1, 0, 1, 1, 0, 1, 0, 0])[:, None]
    d = om.dispatch(idx, 2, C)
    assert list(d.counts) == [4, 4] and list(d.kept) == [2, 2]
    assert list(d.offsets) == [0, 2, 4]
    assert list(d.perm_token) == [1, 4, 0, 2]
    assert list(d.slot_of) == [2, 0, 3, -1, 1, -1, -1, -1]
    # min_capacity raises a small capacity
    assert om.capacity(OracleConfig(T=8, d_model=1, d_ff=1, E=2, k=1,
                                    capacity_factor=0.1, min_capacity=4)) == 4
    assert om.capacity(OracleConfig(T=8, d_model=1, d_ff=1, E=2, k=1)) is None


def test_capacity_hand_example():
    check_capacity_hand_example()


def check_dispatch_invariants(seed=7):
    rng = np.random.default_rng(seed)
    for T, E, k, C in [(100, 8, 2, None), (100, 8, 2, 7), (64, 16, 4, 3), (50, 4, 1, 0),
                       (33, 5, 3, 1)]:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
        d = om.dispatch(idx, E, C)
        flat = idx.reshape(-1)
        # counts by plain counting
        for e in range(E):
            assert d.counts[e] == int(np.sum(flat == e))
        cap = np.inf if C is None else C
        assert np.all(d.kept <= cap) and np.all(d.kept == np.minimum(d.counts, cap))
        assert d.offsets[0] == 0 and np.array_equal(np.diff(d.offsets), d.kept)
        # walk the assignments in t*k+j order with a running counter per expert
        seen = np.zeros(E, np.int64)
        rows_of_e = {e: [] for e in range(E)}
        for a in range(T * k):
            e = flat[a]
            r = seen[e]
            seen[e] += 1
            if r < cap:
                assert d.slot_of[a] == d.offsets[e] + r
                rows_of_e[e].append(a)
            else:
                assert d.slot_of[a] == -1
        # perm_token is a bijection onto the kept assignments, ordered in t*k+j
        kept_slots = d.slot_of[d.slot_of >= 0]
        assert sorted(kept_slots.tolist()) == list(range(int(d.offsets[-1])))
        for e in range(E):
            toks = d.perm_token[d.offsets[e]:d.offsets[e + 1]]
            assert list(toks) == [a // k for a in rows_of_e[e]]


def test_dispatch_invariants():
    check_dispatch_invariants()


# ---------------------------------------------------------------- whole layer
def _brute_forward(cfg, x, w_g, ex, sh, select_bias=None, logit_bias=None):
    """Token by token: route, count earlier assignments of the same expert in
    t*k+j order to decide drops, add w * FFN_e(x_t) (torch MLP), add shared."""
    T, E, k = cfg.T, cfg.E, cfg.k
    l = om.router_logits(x, w_g, logit_bias)
    g = om.gate(l, cfg, select_bias)
    C = om.capacity(cfg)
    seen = [0] * E
    out = np.zeros((T, cfg.d_model))
    for t in range(T):
        for j in range(k):
            e = int(g.idx[t, j])
            r = seen[e]
            seen[e] += 1
            if C is not None and r >= C:
                continue
            out[t] += g.w[t, j] * _torch_ffn(x[t:t + 1], *ex[e])[0]
        for s in range(cfg.n_shared):
            out[t] += _torch_ffn(x[t:t + 1], *sh[s])[0]
    return out


def check_forward_bruteforce(seed=8):
    rng = np.random.default_rng(seed)
    cases = [
        dict(T=24, d_model=8, d_ff=12, E=4, k=2, route=om.ROUTE_SOFTMAX_TOPK),
        dict(T=24, d_model=8, d_ff=12, E=4, k=1, route=om.ROUTE_SOFTMAX_TOPK,
             renorm=False, capacity_factor=1.0),
        dict(T=30, d_model=6, d_ff=10, E=5, k=2, route=om.ROUTE_TOPK_SOFTMAX,
             capacity_factor=1.5),
        dict(T=20, d_model=8, d_ff=8, E=8, k=3, n_shared=1, route=om.ROUTE_BIASED_SOFTMAX),
    ]
    for kw in cases:
        cfg = OracleConfig(**kw)
        x, w_g, ex, sh = _rand_layer(rng, cfg.T, cfg.d_model, cfg.d_ff, cfg.E, cfg.n_shared)
        sb = rng.standard_normal(cfg.E) * 0.01
        lb = rng.standard_normal(cfg.E).astype(np.float32)
        r = om.moe_forward(cfg, x, w_g, lambda e: ex[e], lambda s: sh[s],
                           select_bias=sb, logit_bias=lb)
        want = _brute_forward(cfg, x, w_g, ex, sh, select_bias=sb, logit_bias=lb)
        np.testing.assert_allclose(r.out, want, rtol=1e-11, atol=1e-12)
        # a row subset gives the same rows
        rows = [0, 3, cfg.T - 1]
        rs = om.moe_forward(cfg, x, w_g, lambda e: ex[e], lambda s: sh[s],
                            select_bias=sb, logit_bias=lb, rows=rows)
        np.testing.assert_allclose(rs.out, r.out[rows], rtol=0, atol=1e-13)


def test_forward_bruteforce():
    check_forward_bruteforce()


def check_dropped_tokens_output_zero():
    """Capacity 0 (CF tiny) drops everything: the routed part is exactly 0."""
    rng = np.random.default_rng(9)
    cfg = OracleConfig(T=16, d_model=4, d_ff=6, E=4, k=1, capacity_factor=0.01)
    x, w_g, ex, _ = _rand_layer(rng, 16, 4, 6, 4)
    r = om.moe_forward(cfg, x, w_g, lambda e: ex[e])
    assert r.C == 0 and np.all(r.disp.slot_of == -1) and np.all(r.out == 0)


def test_dropped_tokens_output_zero():
    check_dropped_tokens_output_zero()


def check_router_z_loss():
    """z-loss pins: uniform logits give log(E)^2 exactly; a hand-computed
    two-token case; adding c to every logit of a token moves its log-sum-exp
    by exactly c; the full-layer result carries the same value."""
    for E in (1, 2, 8, 64):
        z = om.router_z_loss(np.zeros((5, E), np.float32))
        assert abs(z - math.log(E) ** 2) < 1e-12, (E, z)
    # token 0: logits 0 and log 3 -> lse = log(1 + 3) = log 4 (log 3 as float32);
    # token 1: two equal logits 1 -> lse = 1 + log 2
    l = np.array([[0.0, math.log(3.0)], [1.0, 1.0]], np.float32)
    lse0 = math.log(1.0 + math.exp(float(l[0, 1])))
    assert abs(lse0 - math.log(4.0)) < 1e-6
    want = (lse0 ** 2 + (1.0 + math.log(2.0)) ** 2) / 2.0
    assert abs(om.router_z_loss(l) - want) < 1e-12, (om.router_z_loss(l), want)
    rng = np.random.default_rng(5)
    a = rng.standard_normal((7, 6)).astype(np.float32)
    c = 2.5
    la = om.router_z_loss(a)
    lse = np.log(np.exp(a.astype(np.float64)).sum(-1))
    assert abs(la - np.mean(lse ** 2)) < 1e-12
    shifted = om.router_z_loss((a + np.float32(c)).astype(np.float32))
    want_shift = np.mean((np.log(np.exp((a + np.float32(c)).astype(np.float64)).sum(-1))) ** 2)
    assert abs(shifted - want_shift) < 1e-9
    assert abs(shifted - np.mean((lse + c) ** 2)) < 1e-5
    cfg = om.OracleConfig(T=7, d_model=4, d_ff=4, E=6, k=2)
    x = rng.standard_normal((7, 4))
    w_g = rng.standard_normal((4, 6)) * 0.5
    ex = {e: (rng.standard_normal((4, 4)), None, rng.standard_normal((4, 4)), None)
          for e in range(6)}
    r = om.moe_forward(cfg, x, w_g, lambda e: ex[e])
    assert abs(r.extra["z_loss"] - om.router_z_loss(r.logits)) == 0.0


def test_router_z_loss():
    check_router_z_loss()


# ---------------------------------------------------------------- Expert Choice
def _ec_brute(col, C):
    """Among all C-subsets of the tokens, the one with the largest logit sum,
    the lexicographically smallest on equal sums (the lower tokens win ties)."""
    best = None
    for sub in itertools.combinations(range(len(col)), C):
        key = (Fraction(0) + sum(Fraction(float(col[t])) for t in sub), [-t for t in sub])
        if best is None or key > best[0]:
            best = (key, sub)
    return list(best[1])


def check_expert_choice_selection(seed=13):
    """Each expert's chosen tokens against subset enumeration (random logits,
    then columns with ties); weights against a hand example: logits (0, log 3)
    give p = (1/4, 3/4)."""
    rng = np.random.default_rng(seed)
    for T, E, C in ((7, 3, 3), (6, 4, 1), (5, 2, 5)):
        l = rng.standard_normal((T, E)).astype(np.float32)
        ec = om.expert_choice(l, C)
        for e in range(E):
            assert list(ec.tokens[e]) == _ec_brute(l[:, e], C), (T, E, C, e)
    l = np.array([[1, 0], [2, 2], [2, 0], [0, 5], [2, 1]], np.float32)
    ec = om.expert_choice(l, 2)
    assert ec.tokens.tolist() == [[1, 2], [1, 3]]
    assert ec.tokens.tolist() == [_ec_brute(l[:, 0], 2), _ec_brute(l[:, 1], 2)]
    l = np.array([[0.0, LN3], [LN3, 0.0]])
    ec = om.expert_choice(l, 1)
    assert ec.tokens.tolist() == [[1], [0]]
    np.testing.assert_allclose(ec.w, [[0.75], [0.75]], rtol=1e-15)
    # selection is on the logits, not on the softmax: token 1 has the larger
    # logit for expert 0 (2 > 1) but the smaller probability (0.27 < 0.73)
    ec = om.expert_choice(np.array([[1.0, 0.0], [2.0, 3.0]]), 1)
    assert ec.tokens[0].tolist() == [1]


def test_expert_choice_selection():
    check_expert_choice_selection()


def check_expert_choice_layer(seed=14):
    """Expert Choice layer pins: every expert processes exactly C tokens;
    f = C/T and aux = alpha * E * C / T; E = 1 with C = T is one dense FFN;
    identical experts with C = T give FFN(x) (the probabilities sum to one);
    W_g = 0 makes every expert take tokens 0..C-1, each with weight 1/E;
    a brute-force layer on tiny inputs."""
    rng = np.random.default_rng(seed)
    T, d, F = 10, 5, 7
    ec_cfg = lambda **kw: _cfg(T=T, d_model=d, d_ff=F, k=1, route=om.ROUTE_EXPERT_CHOICE, **kw)
    x, w_g, ex, _ = _rand_layer(rng, T, d, F, 1)
    r = om.moe_forward(ec_cfg(E=1, capacity_factor=1.0), x, w_g, lambda e: ex[e])
    assert r.C == T
    np.testing.assert_allclose(r.out, _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)
    E = 4
    x, w_g, ex, _ = _rand_layer(rng, T, d, F, E)
    r = om.moe_forward(ec_cfg(E=E, capacity_factor=float(E)), x, w_g, lambda e: ex[0])
    np.testing.assert_allclose(r.out, _torch_ffn(x, *ex[0]), rtol=1e-12, atol=1e-12)
    cfg = ec_cfg(E=E, capacity_factor=1.2, aux_alpha=0.01)
    C = 3                                     # floor(1.2 * 10 / 4)
    r = om.moe_forward(cfg, x, np.zeros_like(w_g), lambda e: ex[0])
    assert r.C == C and r.extra["ec"].tokens.tolist() == [[0, 1, 2]] * E
    assert np.all(r.disp.counts == C) and r.disp.offsets.tolist() == [0, 3, 6, 9, 12]
    np.testing.assert_allclose(r.out[:C], _torch_ffn(x[:C], *ex[0]), rtol=1e-12, atol=1e-12)
    assert np.all(r.out[C:] == 0)
    np.testing.assert_allclose(r.f, np.full(E, C / T), rtol=0, atol=0)
    assert abs(r.aux - 0.01 * E * C / T) < 1e-15
    # brute force: subsets per expert, torch softmax and torch FFNs
    r = om.moe_forward(cfg, x, w_g, lambda e: ex[e])
    l = np.asarray(r.logits)
    p = torch.softmax(torch.as_tensor(l, dtype=torch.float64), dim=-1).numpy()
    want = np.zeros((T, d))
    for e in range(E):
        for t in _ec_brute(l[:, e], C):
            want[t] += p[t, e] * _torch_ffn(x[t:t + 1], *ex[e])[0]
    np.testing.assert_allclose(r.out, want, rtol=1e-12, atol=1e-12)


def test_expert_choice_layer():
    check_expert_choice_layer()


# ---------------------------------------------------------------- planted mistakes
ALL_CHECKS = [check_golden_pages_values, check_selection_bruteforce, check_hand_gate_examples,
              check_softmax_topk_equals_topk_softmax, check_weights_sum_to_one,
              check_softmax_basic, check_router_logits, check_gelu_closed_form,
              check_dense_reductions, check_aux_uniform_router, check_aux_hand_example,
              check_aux_nonnegative_and_argmax, check_capacity_hand_example,
              check_dispatch_invariants, check_forward_bruteforce,
              check_dropped_tokens_output_zero, check_router_z_loss, check_silu_closed_form,
              check_glu_experts, check_expert_choice_selection, check_expert_choice_layer]


def _some_pin_fails():
    failed = []
    for c in ALL_CHECKS:
        try:
            c()
        except (AssertionError, ValueError, IndexError):
            failed.append(c.__name__)
    return failed


def test_all_pins_pass_unplanted():
    assert _some_pin_fails() == []


def _tanh_gelu(v):
    v = np.asarray(v, np.float64)
    return 0.5 * v * (1 + np.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))


def _ffn_transposed(xe, w1, b1, w2, b2, act=om.ACT_GELU):
    # plausible slip: second layer multiplied without the transpose of W2 when
    # d == d_ff would go unnoticed; with d != d_ff this must raise or differ
    h = om.gelu(np.asarray(xe) @ np.asarray(w1).T + (0 if b1 is None else b1))
    return h @ np.asarray(w2).reshape(np.asarray(w2).shape[::-1]) + (0 if b2 is None else b2)


def _select_highest_index_on_ties(score, k):
    s = np.asarray(score, np.float64)
    order = np.argsort(-s[:, ::-1], axis=-1, kind="stable")
    order = s.shape[1] - 1 - order
    m = min(k + 1, s.shape[1])
    top = np.take_along_axis(s, order[:, :m], axis=-1)
    return order[:, :k], np.min(top[:, :-1] - top[:, 1:], axis=-1)


def _capacity_ceil(cfg):
    if cfg.capacity_factor <= 0:
        return None
    return max(int(math.ceil(cfg.capacity_factor * cfg.T / cfg.E)), cfg.min_capacity)


_orig_load_balance = om.load_balance
_orig_expert_ffn = om.expert_ffn
_orig_expert_choice = om.expert_choice


def _ec_highest_token_on_ties(logits, C, override=None):
    l = np.asarray(logits, np.float64)
    T = l.shape[0]
    flipped = _orig_expert_choice(l[::-1], C, override)
    flipped.tokens = np.sort(T - 1 - flipped.tokens, axis=1)
    flipped.p = flipped.p[::-1]
    flipped.w = flipped.p[flipped.tokens, np.arange(l.shape[1])[:, None]]
    return flipped


def _ec_on_softmax(logits, C, override=None):
    p = om.softmax(np.asarray(logits, np.float64))
    r = _orig_expert_choice(p, C, override)
    r.p = p
    r.w = p[r.tokens, np.arange(p.shape[1])[:, None]]
    return r


def _ec_renormalised(logits, C, override=None):
    r = _orig_expert_choice(logits, C, override)
    tot = np.zeros(r.p.shape[0])
    np.add.at(tot, r.tokens.reshape(-1), r.w.reshape(-1))
    r.w = r.w / tot[r.tokens]
    return r


def _silu_as_sigmoid(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


def _swiglu_halves_swapped(xe, w1, b1, w2, b2, act=om.ACT_GELU):
    if act == om.ACT_SWIGLU:
        F = np.asarray(w1).shape[0] // 2
        w1 = np.concatenate([np.asarray(w1)[F:], np.asarray(w1)[:F]])
        if b1 is not None:
            b1 = np.concatenate([np.asarray(b1)[F:], np.asarray(b1)[:F]])
    return _orig_expert_ffn(xe, w1, b1, w2, b2, act=act)


def _z_without_square(logits):
    l = np.asarray(logits, np.float64)
    m = l.max(axis=-1, keepdims=True)
    return float(np.mean(m[:, 0] + np.log(np.exp(l - m).sum(axis=-1))))


def _z_without_max(logits):
    l = np.asarray(logits, np.float64)
    return float(np.mean(np.log(np.exp(l - l.max(axis=-1, keepdims=True)).sum(-1)) ** 2))


@pytest.mark.parametrize("name,patch", [
    ("tanh GELU", ("gelu", _tanh_gelu)),
    ("untransposed W2", ("expert_ffn", _ffn_transposed)),
    ("highest index wins ties", ("select_topk", _select_highest_index_on_ties)),
    ("ceil capacity", ("capacity", _capacity_ceil)),
    ("z-loss not squared", ("router_z_loss", _z_without_square)),
    ("SiLU as the plain sigmoid", ("silu", _silu_as_sigmoid)),
    ("SwiGLU gate and up halves swapped", ("expert_ffn", _swiglu_halves_swapped)),
    ("Expert Choice ties to the highest token", ("expert_choice", _ec_highest_token_on_ties)),
    ("Expert Choice on the softmax", ("expert_choice", _ec_on_softmax)),
    ("Expert Choice weights renormalised per token", ("expert_choice", _ec_renormalised)),
    ("z-loss without the max term", ("router_z_loss", _z_without_max)),
    ("aux without the E factor", ("load_balance",
                                  lambda c, l, p, n: (lambda r: (r[0], r[1], r[2] / c.E))(
                                      _orig_load_balance(c, l, p, n)))),
])
def test_plant_mistake_is_caught(monkeypatch, name, patch):
    attr, fn = patch
    monkeypatch.setattr(om, attr, fn)
    assert _some_pin_fails(), f"planted mistake '{name}' passed every pin"
