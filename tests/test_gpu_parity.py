"""Device parity: the CUDA path through the C ABI against the CPU oracle, on
the same seeded inputs.  Small cases cover every routing form, the capacity
drop, shared experts, biases, ragged tails and several tiles; the full-size
workloads run in the launch configuration the benchmark times, checked on all
tokens for routing/dispatch and on all (or sampled) tokens for the output."""

import numpy as np
import pytest
import torch

from oracle import compare, moe_oracle as om
from sparse_mixture_experts_52_b300 import moe, synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _np(t):
    if t is None:
        return None
    return t.detach().cpu().numpy() if t.dtype not in (torch.bfloat16,) else \
        t.detach().float().cpu().numpy()


def run_forward(cfg, inp):
    layer = moe.MoELayer(cfg, inp, device=DEV)
    r = layer(inp["x"])
    moe.check_status(layer.ws)
    return {k: _np(v) for k, v in r.items()}


def run_steps(cfg, inp):
    """route -> permute -> grouped_ffn -> combine through the four entry points."""
    T, d, E, k, S = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"], cfg.get("n_shared", 0)
    dt = moe.TORCH_DTYPES[cfg["dtype"]]
    yt = moe.y_dtype(cfg)
    ws = moe.new_workspace(cfg, DEV)
    z = lambda shape, t: torch.empty(shape, dtype=t, device=DEV)
    o = dict(logits=z((T, E), torch.float32), topk_idx=z((T, k), torch.int32),
             topk_w=z((T, k), torch.float32), f=z((E,), torch.float32),
             P=z((E,), torch.float32), aux=z((1,), torch.float32),
             z_loss=z((1,), torch.float32), counts=z((E,), torch.int32),
             kept=z((E,), torch.int32), offsets=z((E + 1,), torch.int32),
             perm_token=z((T * k,), torch.int32), slot_of=z((T * k,), torch.int32),
             x_perm=z((T * k, d), dt), y_perm=z((T * k, d), yt), out=z((T, d), dt))
    o["y_shared"] = z((S, T, d), yt) if S else None
    moe.route(cfg, inp["x"], inp["w_g"], o["topk_idx"], o["topk_w"], o["f"], o["P"], o["aux"],
              ws, logit_bias=inp.get("logit_bias"), select_bias=inp.get("select_bias"),
              logits=o["logits"], z_loss=o["z_loss"])
    moe.permute(cfg, inp["x"], o["topk_idx"], o["counts"], o["kept"], o["offsets"],
                o["perm_token"], o["slot_of"], o["x_perm"], ws)
    moe.grouped_ffn(cfg, o["x_perm"], o["offsets"], inp["w1"], inp["w2"], o["y_perm"], ws,
                    b1=inp.get("b1"), b2=inp.get("b2"), x=inp["x"], ws1=inp.get("ws1"),
                    wsb1=inp.get("wsb1"), ws2=inp.get("ws2"), wsb2=inp.get("wsb2"),
                    y_shared=o["y_shared"])
    moe.combine(cfg, o["y_perm"], o["slot_of"], o["topk_w"], o["out"], y_shared=o["y_shared"])
    moe.check_status(ws)
    return {kk: (v if kk in ("x_perm", "y_perm", "out", "y_shared") else _np(v))
            for kk, v in o.items() if v is not None}


def check_steps(cfg, inp, st, rep_ref):
    """Intermediates of the step-wise path against the oracle."""
    ref = compare.run_oracle(cfg, inp, rows=[0])
    if rep_ref.overridden:
        ov = {t: st["topk_idx"][t].astype(np.int64) for t in rep_ref.overridden}
        ref = compare.run_oracle(cfg, inp, rows=[0], idx_override=ov)
    # logits: fp32 sums on the device vs the oracle's float64 sum rounded once.
    # Forward error bound of an fp32 dot product of length d: gamma_d * sum|x_i w_i|
    # (u = 2^-23 allows truncating accumulation), plus the final rounding.
    lg = st["logits"].astype(np.float64)
    x64, wg64 = compare.np64(inp["x"]), compare.np64(inp["w_g"])
    d = cfg["d_model"]
    u = 2.0 ** -23
    bound = (d * u / (1 - d * u)) * (np.abs(x64) @ np.abs(wg64)) + u * np.abs(ref.logits)
    excess = np.abs(lg - ref.logits) - bound
    assert excess.max() <= 0, f"logits beyond the fp32 dot-product bound by {excess.max():.3e}"
    zr = float(ref.extra["z_loss"])
    assert abs(float(st["z_loss"][0]) - zr) <= compare.TOL_Z_REL * abs(zr), "z_loss differs"
    compare.compare_dispatch(ref, st)
    n = int(ref.disp.offsets[-1])
    # x_perm rows are exact copies of x[perm_token]
    xp = st["x_perm"][:n]
    want = inp["x"][torch.as_tensor(ref.disp.perm_token, device=DEV)]
    assert torch.equal(xp, want), "x_perm is not x[perm_token]"
    # y_perm rows are FFN_e of those rows (bf16 / fp32 tolerances)
    experts = compare.LazyExperts(inp["w1"], inp.get("b1"), inp["w2"], inp.get("b2"))
    yp = compare.np64(st["y_perm"][:n])
    x64 = compare.np64(inp["x"])
    for e in range(cfg["E"]):
        a, b = int(ref.disp.offsets[e]), int(ref.disp.offsets[e + 1])
        if a == b:
            continue
        yr = om.expert_ffn(x64[ref.disp.perm_token[a:b]], *experts(e),
                           act=cfg.get("act", om.ACT_GELU))
        rel = np.linalg.norm(yp[a:b] - yr) / max(np.linalg.norm(yr), 1e-30)
        tol = compare.TOL_F32_REL_L2 if cfg["dtype"] == "f32" else compare.TOL_BF16_REL_L2
        assert rel <= tol, f"expert {e}: y_perm rel-L2 {rel:.3e}"


SMALL = {
    "fp32_top2_bias": dict(name="tiny_fp32_top2", T=300, d_model=64, d_ff=96, E=8, k=2,
                           nonzero_bias=True),
    "fp32_warp_router_e24": dict(name="tiny_fp32_top2", T=700, d_model=96, d_ff=64, E=24, k=3,
                                 route="topk_softmax"),
    "switch_cap_small": dict(name="switch_top1_cap", T=1000, d_model=128, d_ff=384, E=16, k=1),
    "switch_cap_renorm": dict(name="switch_top1_cap", T=600, d_model=64, d_ff=128, E=8, k=1,
                              renorm=1, aux_f="topk_count"),
    "mixtral_small_tc_router": dict(name="mixtral_top2", T=600, d_model=256, d_ff=512),
    "mixtral_small_warp_router": dict(name="mixtral_top2", T=200, d_model=256, d_ff=512),
    # the fused tensor-core router: one CTA per 128 tokens (16384 tokens),
    # clusters of 2 with a ragged last tile (8000 tokens), a cluster of 4
    # splitting d = 320 unevenly (E = 16, two 16-byte W_g loads a row), and
    # E = 6 (W_g rows of 12 bytes, element loads)
    "tc_router_no_split": dict(name="mixtral_top2", T=16384, d_model=256, d_ff=128),
    "tc_router_split2_ragged_t": dict(name="mixtral_top2", T=8000, d_model=256, d_ff=128),
    "tc_router_e16_split4_ragged_d": dict(name="mixtral_top2", T=4096, d_model=320, d_ff=128,
                                          E=16, k=4),
    "tc_router_e6_scalar_w": dict(name="mixtral_top2", T=1024, d_model=192, d_ff=128, E=6),
    # the tensor-core router's three launches (transposed W_g, logits GEMM,
    # gating grid) at E = 64 and E = 32
    "tc_router_e64_top1": dict(name="switch_top1_cap", T=1024, d_model=256, d_ff=128, E=64),
    "tc_router_e32_biased": dict(name="deepseek_v3_top8", T=1024, d_model=256, d_ff=128, E=32,
                                 k=4, n_shared=0),
    "softmax_topk_k3_ragged": dict(name="mixtral_top2", route="softmax_topk", T=333,
                                   d_model=200, d_ff=328, E=12, k=3),
    "deepseek_small_e256": dict(name="deepseek_v3_top8", T=256, d_model=128, d_ff=64),
    "deepseek_small_e64_s2": dict(name="deepseek_v3_top8", T=300, d_model=256, d_ff=128,
                                  E=64, k=6, n_shared=2),
    "bf16_bias_shared": dict(name="deepseek_v3_top8", T=300, d_model=128, d_ff=256, E=8, k=2,
                             has_bias=1, nonzero_bias=True),
    "decode_small": dict(name="decode_zipf_top2", T=64, d_model=512, d_ff=1024),
    "cap_min_capacity": dict(name="switch_top1_cap", T=512, d_model=64, d_ff=64, E=16, k=2,
                             capacity_factor=0.25, min_capacity=5, route="softmax_topk",
                             renorm=1, aux_f="topk_count"),
    # expert activations: SiLU, and SwiGLU (gate and up halves in one up-GEMM)
    "silu_small": dict(name="mixtral_top2", T=600, d_model=256, d_ff=512, act="silu"),
    "swiglu_bias_shared_ragged": dict(name="deepseek_v3_top8", T=300, d_model=128, d_ff=200,
                                      E=8, k=2, has_bias=1, nonzero_bias=True, act="swiglu"),
    "swiglu_top1_fused_combine": dict(name="switch_top1_cap", T=1000, d_model=128, d_ff=256,
                                      E=16, k=1, renorm=1, act="swiglu"),
    # raw top-1 gate values (down to 1/E): outputs reach 11x their RMS, so the
    # step-wise path keeps the expert outputs in fp32 (one rounding, in the
    # combine, as the fused path has)
    "swiglu_top1_raw_gate_y_f32": dict(name="switch_top1_cap", T=1000, d_model=128, d_ff=256,
                                       E=16, k=1, renorm=0, act="swiglu", y_f32=1),
    # experts with >= 512 rows each: the CTA-pair GEMM (256-row tiles), with
    # every epilogue, shared experts, biases and ragged d / F
    "pair_gelu_top2": dict(name="mixtral_top2", T=2048, d_model=256, d_ff=512),
    "pair_swiglu_shared_bias": dict(name="deepseek_v3_top8", T=1024, d_model=128, d_ff=256, E=4,
                                    k=2, has_bias=1, nonzero_bias=True, act="swiglu"),
    "pair_top1_fused_combine": dict(name="switch_top1_cap", T=2048, d_model=256, d_ff=512, E=4),
    "pair_y_f32_silu": dict(name="mixtral_top2", T=2048, d_model=128, d_ff=256, E=4, act="silu",
                            y_f32=1),
    "pair_ragged_k3": dict(name="mixtral_top2", route="softmax_topk", T=2048, d_model=200,
                           d_ff=328, E=12, k=3),
    # fp32 expert outputs through moe_forward's own combine (top-2), with a
    # shared expert and biases
    "y_f32_top2_shared_bias": dict(name="deepseek_v3_top8", T=300, d_model=128, d_ff=256, E=8,
                                   k=2, has_bias=1, nonzero_bias=True, y_f32=1),
    "swiglu_fp32_bias": dict(name="tiny_fp32_top2", T=300, d_model=64, d_ff=96, E=8, k=2,
                             nonzero_bias=True, act="swiglu"),
    "silu_fp32": dict(name="tiny_fp32_top2", T=200, d_model=64, d_ff=80, E=4, k=2, act="silu"),
}


def _case(spec):
    spec = dict(spec)
    name = spec.pop("name")
    nz = spec.pop("nonzero_bias", False)
    cfg = synth.workload(name, **spec)
    inp = synth.make_inputs(cfg, device=DEV, nonzero_bias=nz)
    return cfg, inp


@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_case_forward_and_steps(case):
    cfg, inp = _case(SMALL[case])
    fw = run_forward(cfg, inp)
    rep = compare.check_layer(cfg, inp, fw)
    st = run_steps(cfg, inp)
    check_steps(cfg, inp, st, rep)
    assert np.array_equal(st["topk_idx"], fw["topk_idx"])
    if cfg["dtype"] == "bf16" and cfg["k"] == 1 and cfg.get("n_shared", 0) == 0:
        # moe_forward folds the top-1 combine into the down-projection (one
        # rounding fewer than the step-wise path): both meet the tolerance
        rep_st = compare.check_layer(cfg, inp, {"topk_idx": st["topk_idx"], "out": _np(st["out"])})
        print(case, "steps:", rep_st.summary())
    else:
        # the step-wise path and moe_forward run the same kernels in the same order
        assert np.array_equal(_np(st["out"]), fw["out"]), "steps and forward differ"
    print(case, rep.summary())


@pytest.mark.parametrize("name", ["tiny_fp32_top2", "switch_top1_cap", "decode_zipf_top2"])
def test_full_workload_all_tokens(name):
    cfg = synth.workload(name)
    inp = synth.make_inputs(cfg, device=DEV)
    fw = run_forward(cfg, inp)
    rep = compare.check_layer(cfg, inp, fw)
    if name == "switch_top1_cap":
        ref = compare.run_oracle(cfg, inp, rows=[0])
        assert ref.C == 80
    print(name, rep.summary())


def _pick_split(N, row_tiles, sms=148):
    """The tile width and stream-K choice of the library's expert-FFN GEMMs
    (the host-side rule of the tcgen05 grouped GEMM, restated here to find the
    tiles its stream-K tail covers)."""
    wide = 256 if N >= 256 else (128 if N >= 128 else 64)
    if row_tiles * -(-N // wide) >= 8 * sms:
        return wide, True
    return wide, False


def stream_k_tail_tokens(cfg, offsets, perm_token, sms=148):
    """Tokens whose rows lie in the tiles that the up- or down-projection
    splits stream-K (the last waves of a many-wave GEMM): the first and last
    row of every such tile.  A model of the library's schedule: group-major
    tiles, then column block, then 128-row block; whole waves round robin,
    the last one to two waves' tiles split by k-iterations."""
    T, d, F, E, k, S = (cfg["T"], cfg["d_model"], cfg["d_ff"], cfg["E"], cfg["k"],
                        cfg.get("n_shared", 0))
    glu = cfg.get("act", "gelu") == "swiglu"
    n_rows = T * k
    if n_rows >= 512 * E:   # the CTA-pair GEMM: whole tiles only, no stream-K tail
        return []
    rt = max(-(-n_rows // 128) + E // 2, min(E, n_rows)) + S * -(-T // 128)
    rows = [int(offsets[g + 1] - offsets[g]) for g in range(E)] + [T] * S
    toks = set()
    for N_pick, N_out, halve in ((2 * F if glu else F, F, glu), (d, d, False)):
        bn, sk = _pick_split(N_pick, rt, sms)
        if not sk:
            continue
        bno = bn // 2 if halve else bn
        n_tiles = -(-N_out // bno)
        grid = min(sms, 160)
        starts = np.concatenate([[0], np.cumsum([-(-r // 128) * n_tiles for r in rows])])
        total = int(starts[-1])
        waves = total // grid
        dp = (waves - 1) * grid if waves >= 2 else 0
        for t in range(dp, total):
            g = int(np.searchsorted(starts, t, side="right") - 1)
            mt = -(-rows[g] // 128)
            m_blk = (t - int(starts[g])) % mt
            r0, r1 = m_blk * 128, min(m_blk * 128 + 128, rows[g]) - 1
            for r in (r0, r1):
                toks.add(int(perm_token[offsets[g] + r]) if g < E else r)
    return sorted(toks)


@pytest.mark.parametrize("name", ["mixtral_top2", "deepseek_v3_top8", "mixtral_swiglu_top2"])
def test_full_workload_sampled_tokens(name):
    """Routing, statistics and dispatch on every token; the layer output on
    1024 tokens: every token whose rows open or close a tile of the stream-K
    tail (the last waves, whose k-blocks several CTAs share), the rest spread
    evenly over the batch (no capacity limit, so each token's output depends
    only on its own routing)."""
    cfg = synth.workload(name)
    inp = synth.make_inputs(cfg, device=DEV)
    layer = moe.MoELayer(cfg, inp, device=DEV)
    r = layer(inp["x"])
    moe.check_status(layer.ws)
    fw = {k: _np(v) for k, v in r.items()}
    T = cfg["T"]
    ref0 = compare.run_oracle(cfg, inp, rows=[0])
    tail = stream_k_tail_tokens(cfg, ref0.disp.offsets, ref0.disp.perm_token)
    if cfg["T"] * cfg["k"] < 512 * cfg["E"]:
        assert tail, "the full-size workload should split its last waves stream-K"
    if len(tail) > 512:
        tail = [tail[i] for i in np.linspace(0, len(tail) - 1, 512).astype(int)]
    rows = set(tail)
    for t in np.linspace(0, T - 1, 1024).astype(int):
        if len(rows) >= 1024:
            break
        rows.add(int(t))
    rows = sorted(rows)
    rep = compare.check_layer(cfg, inp, fw, rows=rows)
    print(name, f"tail tokens {len(tail)}", rep.summary())
    del layer, inp
    torch.cuda.empty_cache()


def test_determinism_bitwise():
    cfg, inp = _case(SMALL["deepseek_small_e64_s2"])
    a = run_forward(cfg, inp)
    b = run_forward(cfg, inp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("T", [512, 1024])
def test_exact_ties_lowest_index_and_capacity_in_token_order(T):
    """W_g = 0: every logit is exactly 0 on both sides, so every token ties;
    the lowest indices win and the capacity keeps the first tokens (T = 512
    takes the block-per-token router, T = 1024 the tensor-core router with the
    gating in its epilogue)."""
    cfg = synth.workload("switch_top1_cap", T=T, d_model=64, d_ff=64, E=8, k=2,
                         capacity_factor=1.0, renorm=1, aux_f="topk_count")
    inp = synth.make_inputs(cfg, device=DEV)
    inp["w_g"].zero_()
    fw = run_forward(cfg, inp)
    assert np.all(fw["topk_idx"] == np.array([0, 1]))
    assert np.all(fw["topk_w"] == 0.5)
    rep = compare.check_layer(cfg, inp, fw)
    C = int(np.floor(1.0 * T / 8))
    assert list(fw["counts"][:2]) == [T, T]
    st = run_steps(cfg, inp)
    assert list(st["kept"]) == [C, C] + [0] * 6
    sl = st["slot_of"].reshape(T, 2)
    assert np.all(sl[:C] >= 0) and np.all(sl[C:] == -1)
    assert abs(float(fw["aux"][0]) - 2 * 0.01) < 1e-7     # aux = k * alpha (uniform P)
    print(rep.summary())


@pytest.mark.parametrize("mode", ["empty_experts", "all_to_one", "capacity_zero"])
def test_skewed_routing_edges(mode):
    cfg = synth.workload("deepseek_v3_top8", T=400, d_model=128, d_ff=128, E=16, k=2,
                         n_shared=1, route="softmax_topk", select_bias_std=0.0)
    if mode == "capacity_zero":
        cfg["capacity_factor"] = 0.01
    if mode == "all_to_one":
        cfg["capacity_factor"] = 2.0
    inp = synth.make_inputs(cfg, device=DEV)
    lb = torch.zeros(16, device=DEV)
    if mode == "empty_experts":
        lb[3] = -30.0
        lb[9:] = -30.0
    elif mode == "all_to_one":
        lb[5] = 30.0
    inp["logit_bias"] = lb
    fw = run_forward(cfg, inp)
    rep = compare.check_layer(cfg, inp, fw)
    if mode == "empty_experts":
        assert fw["counts"][3] == 0 and np.all(fw["counts"][9:] == 0)
    if mode == "all_to_one":
        assert fw["counts"][5] == 400
    print(mode, rep.summary())


@pytest.mark.parametrize("T", [0, 1, 7])
def test_tiny_token_counts(T):
    cfg = synth.workload("deepseek_v3_top8", T=max(T, 1), d_model=128, d_ff=64, E=32, k=4)
    inp = synth.make_inputs(cfg, device=DEV)
    if T == 0:
        cfg["T"] = 0
        inp["x"] = inp["x"][:0].contiguous()
    fw = run_forward(cfg, inp)
    if T == 0:
        assert np.all(fw["counts"] == 0) and float(fw["aux"][0]) == 0.0
        assert float(fw["z_loss"][0]) == 0.0
        return
    compare.check_layer(cfg, inp, fw)


def test_invalid_argument_enqueues_nothing():
    cfg = synth.workload("tiny_fp32_top2")
    inp = synth.make_inputs(cfg, device=DEV)
    layer = moe.MoELayer(cfg, inp, device=DEV)
    bad = dict(cfg, k=9)
    with pytest.raises(moe.MoEError) as ei:
        moe.forward(bad, inp["x"], inp["w_g"], inp["w1"], inp["w2"], layer.out, layer.ws)
    assert ei.value.status in (1,)
    moe.check_status(layer.ws)


def test_out_of_range_expert_index_is_dropped_and_reported():
    """moe_permute takes caller-supplied indices: one outside [0, E), or one
    repeated in its token's row, drops that assignment (slot -1), the others
    are dispatched as usual, and the status word reports MOE_ERR_INVALID_ARG."""
    cfg = synth.workload("switch_top1_cap", T=96, d_model=64, d_ff=64, E=8, k=2,
                         capacity_factor=0.0, renorm=1, aux_f="topk_count")
    T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
    inp = synth.make_inputs(cfg, device=DEV)
    g = torch.Generator().manual_seed(3)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    idx[5, 1] = E + 3
    idx[40, 0] = -1
    idx[60, 1] = idx[60, 0]          # a repeated expert: the second occurrence drops
    idx = idx.to(DEV)
    ws = moe.new_workspace(cfg, DEV)
    z = lambda shape, t: torch.empty(shape, dtype=t, device=DEV)
    o = dict(counts=z((E,), torch.int32), kept=z((E,), torch.int32),
             offsets=z((E + 1,), torch.int32), perm_token=z((T * k,), torch.int32),
             slot_of=z((T * k,), torch.int32), x_perm=z((T * k, d), torch.bfloat16))
    moe.permute(cfg, inp["x"], idx, o["counts"], o["kept"], o["offsets"], o["perm_token"],
                o["slot_of"], o["x_perm"], ws)
    with pytest.raises(moe.MoEError) as ei:
        moe.check_status(ws)
    assert ei.value.status == 1
    moe.check_status(ws)          # the status word was cleared by the read
    slot = o["slot_of"].cpu().view(T, k)
    assert slot[5, 1] == -1 and slot[40, 0] == -1 and slot[60, 1] == -1 and slot[60, 0] >= 0
    good = idx.cpu().clone()
    good[5, 1] = -1
    good[40, 0] = -1
    good[60, 1] = -1
    want = torch.bincount(good[good >= 0].long(), minlength=E)
    assert torch.equal(o["counts"].cpu(), want.to(torch.int32))
    assert int(o["offsets"][-1]) == T * k - 3
    assert int((slot >= 0).sum()) == T * k - 3
    # every kept assignment has a slot of its own, and perm_token inverts it
    kept = slot[slot >= 0]
    assert len(set(kept.tolist())) == kept.numel()
    pt = o["perm_token"].cpu()
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                assert int(pt[slot[t, j]]) == t


# ---------------------------------------------------------------- Expert Choice
def run_steps_ec(cfg, inp):
    """route -> permute -> grouped_ffn -> combine through the Expert Choice
    entry points."""
    T, d, E, S = cfg["T"], cfg["d_model"], cfg["E"], cfg.get("n_shared", 0)
    C = moe.expert_capacity(cfg)
    dt = moe.TORCH_DTYPES[cfg["dtype"]]
    yt = moe.y_dtype(cfg)
    ws = moe.new_workspace(cfg, DEV)
    z = lambda shape, t: torch.empty(shape, dtype=t, device=DEV)
    o = dict(logits=z((T, E), torch.float32), topk_idx=z((E, C), torch.int32),
             topk_w=z((E, C), torch.float32), ec_slot=z((E, T), torch.int32),
             f=z((E,), torch.float32), P=z((E,), torch.float32), aux=z((1,), torch.float32),
             z_loss=z((1,), torch.float32), offsets=z((E + 1,), torch.int32),
             x_perm=z((E * C, d), dt), y_perm=z((E * C, d), yt), out=z((T, d), dt))
    o["y_shared"] = z((S, T, d), yt) if S else None
    moe.route_expert_choice(cfg, inp["x"], inp["w_g"], o["topk_idx"], o["topk_w"], o["ec_slot"],
                            o["f"], o["P"], o["aux"], ws, logit_bias=inp.get("logit_bias"),
                            logits=o["logits"], z_loss=o["z_loss"])
    moe.permute_expert_choice(cfg, inp["x"], o["topk_idx"], o["offsets"], o["x_perm"])
    moe.grouped_ffn(cfg, o["x_perm"], o["offsets"], inp["w1"], inp["w2"], o["y_perm"], ws,
                    b1=inp.get("b1"), b2=inp.get("b2"), x=inp["x"], ws1=inp.get("ws1"),
                    wsb1=inp.get("wsb1"), ws2=inp.get("ws2"), wsb2=inp.get("wsb2"),
                    y_shared=o["y_shared"])
    moe.combine_expert_choice(cfg, o["y_perm"], o["ec_slot"], o["topk_w"], o["out"],
                              y_shared=o["y_shared"])
    moe.check_status(ws)
    return {kk: (v if kk in ("x_perm", "y_perm", "y_shared") else _np(v))
            for kk, v in o.items() if v is not None}


def check_steps_ec(cfg, inp, st, fw):
    """Step-wise Expert Choice path: the same selection, slot table, rows and
    output as moe_forward (same kernels, same order), and the slot table is
    the inverse of the token lists."""
    E, T = cfg["E"], cfg["T"]
    C = moe.expert_capacity(cfg)
    assert np.array_equal(st["topk_idx"], fw["topk_idx"])
    assert np.array_equal(st["topk_w"], fw["topk_w"])
    assert np.array_equal(st["offsets"], np.arange(E + 1) * C)
    want = np.full((E, T), -1, np.int64)
    for e in range(E):
        want[e, st["topk_idx"][e]] = e * C + np.arange(C)
    assert np.array_equal(st["ec_slot"], want), "slot table is not the inverse of the lists"
    xp = st["x_perm"]
    assert torch.equal(xp, inp["x"][torch.as_tensor(st["topk_idx"].reshape(-1), device=DEV).long()])
    assert np.array_equal(st["out"], fw["out"]), "steps and forward differ"
    for k in ("f", "P", "aux", "z_loss"):
        assert np.array_equal(st[k], fw[k]), k


EC_SMALL = {
    "ec_bf16_ragged": dict(name="switch_expert_choice", T=1000, d_model=128, d_ff=256, E=16),
    "ec_fp32_bias": dict(name="tiny_fp32_top2", T=300, d_model=64, d_ff=96, E=8,
                         route="expert_choice", capacity_factor=1.5, nonzero_bias=True),
    "ec_shared_e64_swiglu": dict(name="deepseek_v3_top8", T=600, d_model=128, d_ff=128, E=64,
                                 route="expert_choice", capacity_factor=4.0, act="swiglu",
                                 select_bias_std=0.0),
    "ec_shared_y_f32": dict(name="deepseek_v3_top8", T=400, d_model=128, d_ff=128, E=16,
                            route="expert_choice", capacity_factor=2.0, select_bias_std=0.0,
                            y_f32=1),
    "ec_argmax_f_min_capacity": dict(name="switch_expert_choice", T=256, d_model=64, d_ff=64,
                                     E=8, capacity_factor=0.01, min_capacity=5,
                                     aux_f="argmax"),
    "ec_every_token": dict(name="switch_expert_choice", T=200, d_model=64, d_ff=64, E=4,
                           capacity_factor=4.0),
    # columns of 6000 tokens (16 in registers per thread) and of 9000 tokens
    # (beyond the register-resident select: the column is streamed)
    "ec_t6000": dict(name="switch_expert_choice", T=6000, d_model=64, d_ff=64, E=8,
                     capacity_factor=1.0),
    "ec_t9000_streamed": dict(name="switch_expert_choice", T=9000, d_model=64, d_ff=64, E=4,
                              capacity_factor=0.5),
}


@pytest.mark.parametrize("case", sorted(EC_SMALL))
def test_expert_choice_small(case):
    cfg, inp = _case(EC_SMALL[case])
    fw = run_forward(cfg, inp)
    rep = compare.check_layer(cfg, inp, fw)
    st = run_steps_ec(cfg, inp)
    check_steps_ec(cfg, inp, st, fw)
    C = moe.expert_capacity(cfg)
    assert fw["topk_idx"].shape == (cfg["E"], C)
    print(case, "C =", C, rep.summary())


def test_expert_choice_ties_and_empty_capacity():
    """W_g = 0: every logit is 0, so every expert takes tokens 0..C-1 with
    weight 1/E.  A capacity of 0 takes nothing: the output is the shared
    expert alone."""
    cfg = synth.workload("switch_expert_choice", T=300, d_model=64, d_ff=64, E=8,
                         capacity_factor=1.0)
    inp = synth.make_inputs(cfg, device=DEV)
    inp["w_g"].zero_()
    fw = run_forward(cfg, inp)
    C = moe.expert_capacity(cfg)
    assert C == 37
    assert np.array_equal(fw["topk_idx"], np.tile(np.arange(C), (8, 1)))
    assert np.all(fw["topk_w"] == np.float32(1 / 8))
    compare.check_layer(cfg, inp, fw)
    cfg = synth.workload("switch_expert_choice", T=100, d_model=64, d_ff=64, E=8,
                         capacity_factor=0.05, n_shared=1)
    inp = synth.make_inputs(cfg, device=DEV)
    assert moe.expert_capacity(cfg) == 0
    fw = run_forward(cfg, inp)
    assert np.all(fw["counts"] == 0)
    compare.check_layer(cfg, inp, fw)


def test_expert_choice_full_workload():
    cfg = synth.workload("switch_expert_choice")
    inp = synth.make_inputs(cfg, device=DEV)
    fw = run_forward(cfg, inp)
    rep = compare.check_layer(cfg, inp, fw)
    assert moe.expert_capacity(cfg) == 128
    print("switch_expert_choice", rep.summary())


def test_streamed_layer_overlapping_copies_match_direct_calls():
    """StreamedMoELayer runs the copies of neighbouring calls on their own
    streams; every call's host output must equal a direct call on the same
    tokens, bit for bit (five calls: both graphed layers are reused)."""
    cfg = synth.workload("switch_top1_cap", T=1000, d_model=128, d_ff=256, E=16)
    inp = synth.make_inputs(cfg, device=DEV)
    ref_layer = moe.MoELayer(cfg, inp, device=DEV)
    s = moe.StreamedMoELayer(cfg, inp, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(5)
    xs = [torch.randn((cfg["T"], cfg["d_model"]), generator=g).to(torch.bfloat16).pin_memory()
          for _ in range(5)]
    outs = [torch.empty((cfg["T"], cfg["d_model"]), dtype=torch.bfloat16).pin_memory()
            for _ in range(5)]
    auxs = [torch.empty((1,), dtype=torch.float32).pin_memory() for _ in range(5)]
    for x, o, a in zip(xs, outs, auxs):
        s.submit(x, o, a)
    s.synchronize()
    for x, o, a in zip(xs, outs, auxs):
        r = ref_layer(x.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(o, r["out"].cpu())
        assert torch.equal(a, r["aux"].cpu())
