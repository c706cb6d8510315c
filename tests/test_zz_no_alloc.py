"""moe_permute_noalloc: the dispatch step for callers that cannot allocate
device memory.

Some hosts own every device allocation through their own pool, or forbid
cudaMalloc on a latency path (it may synchronise the device).  For them the
library offers moe_permute_noalloc, which keeps its rank scratch in a fixed
array inside the library instead of a caller workspace.  These tests call it
through the C ABI and check that it gives exactly what moe_permute gives
(integer and copy work: bit for bit), on consecutive calls that share the
array.  The file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

from sparse_mixture_experts_52_b300 import moe, synth

DEV = "cuda"


def _route(cfg, inp):
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    ws = moe.new_workspace(cfg, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    f = torch.empty((E,), dtype=torch.float32, device=DEV)
    P = torch.empty((E,), dtype=torch.float32, device=DEV)
    aux = torch.empty((1,), dtype=torch.float32, device=DEV)
    moe.route(cfg, inp["x"], inp["w_g"], idx, w, f, P, aux, ws,
              logit_bias=inp.get("logit_bias"), select_bias=inp.get("select_bias"))
    return idx, ws


def _outputs(cfg):
    T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
    dt = moe.TORCH_DTYPES[cfg["dtype"]]
    # sentinel fill so that an entry the call forgot to write cannot match
    z = lambda shape, t: torch.full(shape, -7, dtype=t, device=DEV)
    return dict(counts=z((E,), torch.int32), kept=z((E,), torch.int32),
                offsets=z((E + 1,), torch.int32), perm_token=z((T * k,), torch.int32),
                slot_of=z((T * k,), torch.int32), x_perm=z((T * k, d), dt))


def _check_same(cfg, a, b):
    for key in ("counts", "kept", "offsets", "slot_of"):
        assert torch.equal(a[key], b[key]), key
    n = int(a["offsets"][-1])
    assert torch.equal(a["perm_token"][:n], b["perm_token"][:n]), "perm_token"
    assert torch.equal(a["x_perm"][:n], b["x_perm"][:n]), "x_perm"


CASES = [
    # Switch-style top-1 with a capacity cut (drops happen)
    dict(name="switch_top1_cap", T=2048, d_model=256, d_ff=128, E=32, k=1),
    # fine-grained top-6 over 64 experts: more assignments than the first case
    dict(name="deepseek_v3_top8", T=1500, d_model=128, d_ff=64, E=64, k=6,
         capacity_factor=2.0),
]


@pytest.mark.gpu
def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    prepared = []
    for spec in CASES:
        spec = dict(spec)
        cfg = synth.workload(spec.pop("name"), **spec)
        inp = synth.make_inputs(cfg, device=DEV)
        idx, ws = _route(cfg, inp)
        ref = _outputs(cfg)
        moe.permute(cfg, inp["x"], idx, ref["counts"], ref["kept"], ref["offsets"],
                    ref["perm_token"], ref["slot_of"], ref["x_perm"], ws)
        prepared.append((cfg, inp, idx, ref))
    torch.cuda.synchronize()
    # consecutive calls share the fixed array: A, B, then A again
    for cfg, inp, idx, ref in prepared + prepared[:1]:
        got = _outputs(cfg)
        moe.permute_noalloc(cfg, inp["x"], idx, got["counts"], got["kept"], got["offsets"],
                            got["perm_token"], got["slot_of"], got["x_perm"])
        torch.cuda.synchronize()
        _check_same(cfg, ref, got)
        if cfg["capacity_factor"] > 0 and cfg["k"] == 1:
            assert int((got["slot_of"] < 0).sum()) > 0, "the capacity case should drop"


def test_noalloc_permute_rejects_sizes_beyond_its_array():
    """Host-side check, no GPU work: T*k above the fixed array's size is
    rejected with MOE_ERR_UNSUPPORTED before anything is enqueued."""
    cfg = synth.workload("deepseek_v3_top8", T=moe.PERMUTE_NOALLOC_MAX_ASSIGNMENTS // 8 + 1,
                         d_model=64, d_ff=64, E=16, k=8, n_shared=0)
    c = moe.make_config(cfg)
    s = moe.lib().moe_permute_noalloc(ctypes.byref(c), 1, 1, 1, 1, 1, 1, 1, 1, None)
    assert s == 2, moe.status_string(s)
    ok = synth.workload("deepseek_v3_top8", T=moe.PERMUTE_NOALLOC_MAX_ASSIGNMENTS // 8,
                        d_model=64, d_ff=64, E=16, k=8, n_shared=0)
    c = moe.make_config(ok)
    # at the limit the size check passes and the null counts pointer is what fails
    s = moe.lib().moe_permute_noalloc(ctypes.byref(c), 1, 1, None, 1, 1, 1, 1, 1, None)
    assert s == 1, moe.status_string(s)
    # the per-chunk expert counts (ceil(T/32) * E entries) have a limit of their own
    chunks = moe.PERMUTE_NOALLOC_MAX_CHUNK_COUNTS // 256
    for T, want in ((32 * chunks, 1), (32 * chunks + 1, 2)):
        cfg = synth.workload("deepseek_v3_top8", T=T, d_model=64, d_ff=64, E=256, k=1,
                             n_shared=0)
        c = moe.make_config(cfg)
        s = moe.lib().moe_permute_noalloc(ctypes.byref(c), 1, 1, None, 1, 1, 1, 1, 1, None)
        assert s == want, (T, moe.status_string(s))
