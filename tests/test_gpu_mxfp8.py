"""MX FP8 experts on the device against the oracle's MX quantiser and layer.

The packing entry point is checked bit for bit against the oracle's codes and
scale bytes (integer work); the layer with MX FP8 experts is checked against
the oracle layer that quantises the same operands the same way, within the
bf16 layer tolerances."""

import numpy as np
import pytest
import torch

from oracle import compare, mxfp8 as mx
from sparse_mixture_experts_52_b300 import moe, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def packed_reference(w: np.ndarray, glu: bool):
    """The documented packed layout, built from the oracle's quantiser: codes
    [G, N, K], then 512-byte scale blocks (g, k / 128, n / 128) with the scale
    of row n, k-block j at byte 16 (n % 32) + 4 ((n % 128) / 32) + j, then
    4 KB tile records (g, k / 128, n / 256): blocks 2t and 2t + 1 four times
    each (zeros past the last block)."""
    G, N, K = w.shape
    codes = np.empty((G, N, K), np.uint8)
    sf = np.zeros(G * N * K // 32, np.uint8)
    KS, NB = K // 128, N // 128
    for g in range(G):
        rows = w[g]
        if glu:   # packed row 128 t + i: gate row 64 t + i, or up row F + 64 t + i - 64
            F = N // 2
            order = [64 * (p // 128) + (p % 128) if p % 128 < 64 else F + 64 * (p // 128) + (p % 128) - 64
                     for p in range(N)]
            rows = rows[order]
        c, s = mx.quantize(rows)
        codes[g] = c
        n = np.arange(N)[:, None]
        kb = np.arange(K // 32)[None, :]
        off = ((g * KS + kb // 4) * NB + n // 128) * 512 + (n % 32) * 16 + ((n % 128) // 32) * 4 + kb % 4
        sf[off] = s
    NT = (NB + 1) // 2
    blocks = sf.reshape(G, KS, NB, 512)
    tiles = np.zeros((G, KS, NT, 8, 512), np.uint8)
    for t in range(NT):
        for r in range(8):
            b = 2 * t + r // 4
            if b < NB:
                tiles[:, :, t, r] = blocks[:, :, b]
    return codes, np.concatenate([sf, tiles.reshape(-1)])


@pytest.mark.parametrize("glu", [False, True])
def test_weight_packing_is_bit_exact(glu):
    g = torch.Generator(device=DEV).manual_seed(4)
    # N / 128 odd (dense): the last tile record's second block is zeros
    G, N, K = 3, (512 if glu else 640), 384
    w = (torch.randn((G, N, K), generator=g, device=DEV) *
         torch.exp2(torch.randint(-6, 6, (G, N, 1), generator=g, device=DEV).float())).to(torch.bfloat16)
    w[0, 5, 32:64] = 0          # an all-zero block
    w[1, 7, :32] = 448.0 * 2.0 ** -3
    packed = moe.quantize_mxfp8(w, glu=glu)
    torch.cuda.synchronize()
    codes_ref, sf_ref = packed_reference(w.float().cpu().numpy(), glu)
    got = packed.cpu().numpy()
    n = G * N * K
    assert np.array_equal(got[:n].reshape(G, N, K), codes_ref), "e4m3 codes differ"
    assert np.array_equal(got[n:], sf_ref), "scale bytes differ"


def _layer(spec):
    spec = dict(spec)
    name = spec.pop("name")
    nz = spec.pop("nonzero_bias", False)
    cfg = synth.workload(name, experts="mxfp8", **spec)
    inp = synth.make_inputs(cfg, device=DEV, nonzero_bias=nz)
    return cfg, inp


def run_forward(cfg, inp):
    layer = moe.MoELayer(cfg, inp, device=DEV)
    r = layer(inp["x"])
    moe.check_status(layer.ws)
    return {k: _np(v) for k, v in r.items()}, layer


def run_steps(cfg, inp, layer):
    """route -> permute -> grouped FFN (MX experts, the bf16 x_perm quantised
    inside) -> combine through the step entry points."""
    T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
    ws = moe.new_workspace(cfg, DEV)
    z = lambda shape, t: torch.empty(shape, dtype=t, device=DEV)
    yt = moe.y_dtype(cfg)
    o = dict(topk_idx=z((T, k), torch.int32), topk_w=z((T, k), torch.float32),
             f=z((E,), torch.float32), P=z((E,), torch.float32), aux=z((1,), torch.float32),
             counts=z((E,), torch.int32), kept=z((E,), torch.int32),
             offsets=z((E + 1,), torch.int32), perm_token=z((T * k,), torch.int32),
             slot_of=z((T * k,), torch.int32), x_perm=z((T * k, d), torch.bfloat16),
             y_perm=z((T * k, d), yt), out=z((T, d), torch.bfloat16))
    moe.route(cfg, inp["x"], inp["w_g"], o["topk_idx"], o["topk_w"], o["f"], o["P"], o["aux"], ws,
              logit_bias=inp.get("logit_bias"), select_bias=inp.get("select_bias"))
    moe.permute(cfg, inp["x"], o["topk_idx"], o["counts"], o["kept"], o["offsets"],
                o["perm_token"], o["slot_of"], o["x_perm"], ws)
    moe.grouped_ffn(cfg, o["x_perm"], o["offsets"], layer.w["w1"], layer.w["w2"], o["y_perm"],
                    ws, b1=inp.get("b1"), b2=inp.get("b2"))
    moe.combine(cfg, o["y_perm"], o["slot_of"], o["topk_w"], o["out"])
    moe.check_status(ws)
    return {kk: _np(v) for kk, v in o.items()}


SMALL = {
    "top2_gelu": dict(name="mixtral_top2", T=600, d_model=256, d_ff=512),
    "top2_silu_bias": dict(name="mixtral_top2", T=300, d_model=128, d_ff=384, act="silu",
                           has_bias=1, nonzero_bias=True),
    "top2_swiglu": dict(name="mixtral_top2", T=500, d_model=256, d_ff=256, act="swiglu"),
    "top1_capacity_fused_combine": dict(name="switch_top1_cap", T=1000, d_model=256, d_ff=512,
                                        E=16),
    "top8_biased_e64": dict(name="deepseek_v3_top8", T=256, d_model=256, d_ff=128, E=64,
                            n_shared=0),
    "top2_y_f32": dict(name="mixtral_top2", T=300, d_model=128, d_ff=256, y_f32=1),
    # many waves: the stream-K tail of both projections
    "stream_k_tail": dict(name="mixtral_top2", T=4096, d_model=256, d_ff=4096),
    # experts of >= 512 rows: the block-scaled CTA-pair GEMM (256 x 256 tiles)
    "pair_top2_gelu": dict(name="mixtral_top2", T=2048, d_model=256, d_ff=512),
    "pair_swiglu": dict(name="mixtral_top2", T=2048, d_model=256, d_ff=256, E=4,
                        act="swiglu"),
    "pair_top1_fused_combine": dict(name="switch_top1_cap", T=2048, d_model=256, d_ff=512, E=4),
    "pair_silu_bias_y_f32": dict(name="mixtral_top2", T=2048, d_model=256, d_ff=256, E=4,
                                 act="silu", has_bias=1, nonzero_bias=True, y_f32=1),
    "pair_swiglu_bias_long_k": dict(name="mixtral_top2", T=1536, d_model=512, d_ff=1024, E=4,
                                    act="swiglu", has_bias=1, nonzero_bias=True),
    # many rows but weight rows not whole 256-row tiles: the single-CTA kernel
    "many_rows_ragged_n": dict(name="mixtral_top2", T=2048, d_model=128, d_ff=384, E=4),
}


@pytest.mark.parametrize("case", sorted(SMALL))
def test_mx_layer_against_the_quantising_oracle(case):
    cfg, inp = _layer(SMALL[case])
    fw, layer = run_forward(cfg, inp)
    rows = None
    if cfg["T"] > 1000:
        rows = sorted(set(np.linspace(0, cfg["T"] - 1, 512).astype(int).tolist()))
    rep = compare.check_layer(cfg, inp, fw, rows=rows)
    st = run_steps(cfg, inp, layer)
    assert np.array_equal(st["topk_idx"], fw["topk_idx"])
    if cfg["k"] == 1:
        # the whole-layer pass folds the top-1 combine into the down-projection
        rep_st = compare.check_layer(cfg, inp, {"topk_idx": st["topk_idx"], "out": st["out"]},
                                     rows=rows)
        print(case, "steps:", rep_st.summary())
    else:
        # the step-wise path quantises the same rows into the same layout
        assert np.array_equal(st["out"], fw["out"]), "steps and forward differ"
    print(case, rep.summary())


def test_mx_full_mixtral_sampled_tokens():
    """The Mixtral-shaped layer with MX FP8 experts (CTA pairs): routing on
    every token, the output on 256 tokens spread over the batch."""
    cfg = synth.workload("mixtral_top2_mxfp8")
    inp = synth.make_inputs(cfg, device=DEV)
    fw, layer = run_forward(cfg, inp)
    rows = sorted(set(np.linspace(0, cfg["T"] - 1, 256).astype(int).tolist()))
    rep = compare.check_layer(cfg, inp, fw, rows=rows)
    print("mixtral_top2_mxfp8", rep.summary())
    del layer, inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["switch_top1_cap_mxfp8", "decode_zipf_top2_mxfp8"])
def test_mx_full_workload_all_tokens(name):
    cfg = synth.workload(name)
    inp = synth.make_inputs(cfg, device=DEV)
    fw, layer = run_forward(cfg, inp)
    rep = compare.check_layer(cfg, inp, fw)
    print(name, rep.summary())
    del layer, inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode,T", [("empty_experts", 2048), ("all_to_one", 2048),
                                    ("empty_experts", 300)])
def test_mx_skewed_routing(mode, T):
    """Skewed routing on the MX FP8 kernels: empty experts between busy ones
    (zero-row groups among the 256-row aligned group offsets) and one expert
    taking every token; T = 2048 runs the CTA-pair GEMM, T = 300 the
    single-CTA one."""
    cfg = synth.workload("mixtral_top2", experts="mxfp8", T=T, d_model=256, d_ff=256, E=4)
    inp = synth.make_inputs(cfg, device=DEV)
    lb = torch.zeros(4, device=DEV)
    if mode == "empty_experts":
        lb[1] = -30.0
        lb[3] = -30.0
    else:
        lb[2] = 30.0
    inp["logit_bias"] = lb
    fw, layer = run_forward(cfg, inp)
    rows = None if T <= 1000 else sorted(set(np.linspace(0, T - 1, 512).astype(int).tolist()))
    rep = compare.check_layer(cfg, inp, fw, rows=rows)
    if mode == "empty_experts":
        assert fw["counts"][1] == 0 and fw["counts"][3] == 0
    else:
        assert fw["counts"][2] == T
    print(mode, T, rep.summary())
