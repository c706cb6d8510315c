"""Host-only checks of the C-ABI library: it loads, exports every entry point
include/moe.h declares, and validates arguments without touching a GPU."""

import ctypes
import os
import re

import pytest

from sparse_mixture_experts_52_b300 import moe, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^(?:moe_status|const char\*)\s+(moe_\w+)\s*\(", text, re.M)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from sparse_mixture_experts_52_b300 import build
        build.build()
    return moe.lib()


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ("moe_workspace_size", "moe_workspace_init", "moe_route", "moe_permute",
              "moe_grouped_ffn", "moe_combine", "moe_forward", "moe_check_status",
              "moe_status_string"):
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), f"{n} declared in moe.h but not exported"


def test_config_struct_layout(lib):
    # 15 four-byte fields, no padding
    assert ctypes.sizeof(moe.Config) == 68
    assert moe.Config.capacity_factor.offset == 24
    assert moe.Config.aux_f.offset == 52
    assert moe.Config.act.offset == 56
    assert moe.Config.y_f32.offset == 60
    assert moe.Config.expert_fmt.offset == 64


def test_expert_output_type_flag_is_validated(lib):
    n = ctypes.c_size_t(0)
    sizes = {}
    for y, want in ((0, 0), (1, 0), (2, 1), (-1, 1)):
        c = moe.make_config(synth.workload("mixtral_top2", T=256, y_f32=y))
        assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == want, y
        sizes[y] = n.value
    # fp32 expert outputs take twice the bytes of the bf16 ones in the workspace
    assert sizes[1] > sizes[0]


def test_activation_value_is_validated(lib):
    for act, want in ((0, 0), (1, 0), (2, 0), (3, 1), (-1, 1)):
        c = moe.make_config(synth.workload("tiny_fp32_top2", act=act))
        n = ctypes.c_size_t(0)
        assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == want, act


def test_status_strings(lib):
    for s in range(6):
        assert moe.status_string(s)
    assert moe.status_string(0) == "ok"


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_workspace_size_of_every_workload(lib, name):
    cfg = synth.workload(name)
    n = moe.workspace_size(cfg)
    T, d, F, k, S = cfg["T"], cfg["d_model"], cfg["d_ff"], cfg["k"], cfg["n_shared"]
    eb = 2 if cfg["dtype"] == "bf16" else 4
    # x_perm + H + Y must fit
    assert n >= (T * k * d + (T * k + S * T) * F + T * k * d) * eb
    # MX FP8 experts add codes and scales of the rows at 128-row aligned offsets
    # MX codes and scales of x and h at 256-row aligned expert offsets
    mx = (T * k + 256 * cfg["E"] + 256) * (d + F) * 33 // 32 if cfg.get("experts") == "mxfp8" else 0
    assert n < 4 * (T * k * d + (T * k + S * T) * F + T * k * d) * eb + mx + (1 << 24)


@pytest.mark.parametrize("field,value,status", [
    ("E", 0, 1), ("E", 257, 1), ("k", 0, 1), ("k", 9, 1), ("T", -1, 1),
    ("d_model", 0, 1), ("n_shared", 5, 1), ("route", 3, 1), ("dtype", 2, 1),
    ("aux_f", 2, 1), ("renorm", 2, 1), ("min_capacity", -1, 1),
    ("d_model", 100, 2), ("d_ff", 36, 2),
])
def test_invalid_configs_are_rejected_on_the_host(lib, field, value, status):
    cfg = synth.workload("mixtral_top2", T=16, d_model=64, d_ff=128, k=2, E=8)
    cfg[field] = value
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_size(cfg)
    assert ei.value.status == status


def test_fp32_wide_router_unsupported(lib):
    cfg = synth.workload("tiny_fp32_top2", E=128)
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_size(cfg)
    assert ei.value.status == 2


def test_missing_workspace_is_rejected_before_any_launch(lib):
    cfg = synth.workload("tiny_fp32_top2")
    c = moe.make_config(cfg)
    # no CUDA call happens: the workspace check fails first
    s = lib.moe_route(ctypes.byref(c), 1, 1, None, None, None, 1, 1, 1, 1, 1, None, None, 0,
                      None)
    assert s == 3
    big = moe.workspace_size(cfg)
    s = lib.moe_forward(ctypes.byref(c), 1, 1, None, None, 1, 1, 1, 1, None, None, None, None,
                        1, None, None, None, None, None, None, None, 256, big - 1, None)
    assert s == 3  # too small
    s = lib.moe_forward(ctypes.byref(c), 1, 1, None, None, 1, 1, 1, 1, None, None, None, None,
                        1, None, None, None, None, None, None, None, 257, big, None)
    assert s == 3  # misaligned


def test_null_required_pointers_rejected(lib):
    cfg = synth.workload("tiny_fp32_top2")
    c = moe.make_config(cfg)
    big = moe.workspace_size(cfg)
    # out == NULL
    s = lib.moe_forward(ctypes.byref(c), 1, 1, None, None, 1, 1, 1, 1, None, None, None, None,
                        None, None, None, None, None, None, None, None, 256, big, None)
    assert s == 1
    # missing expert biases while has_bias = 1
    s = lib.moe_forward(ctypes.byref(c), 1, 1, None, None, 1, None, 1, None, None, None, None,
                        None, 1, None, None, None, None, None, None, None, 256, big, None)
    assert s == 1
    s = lib.moe_combine(ctypes.byref(c), None, 1, 1, None, 1, None)
    assert s == 1


def test_expert_choice_host_checks(lib):
    """Expert Choice needs a capacity; the top-k and Expert Choice entry points
    refuse each other's configurations; moe_expert_capacity gives C."""
    ec = synth.workload("switch_expert_choice")
    assert moe.expert_capacity(ec) == 128                       # floor(2.0 * 4096 / 64)
    assert moe.expert_capacity(dict(ec, capacity_factor=100.0)) == 4096   # at most T
    assert moe.expert_capacity(dict(ec, capacity_factor=0.001, min_capacity=7)) == 7
    assert moe.expert_capacity(synth.workload("switch_top1_cap")) == 80
    assert moe.expert_capacity(synth.workload("mixtral_top2")) == -1   # no limit
    n = ctypes.c_size_t(0)
    bad = moe.make_config(dict(ec, capacity_factor=0.0))
    assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1
    c = moe.make_config(ec)
    big = moe.workspace_size(ec)
    # top-k entry points refuse an Expert Choice configuration (nothing enqueued)
    s = lib.moe_route(ctypes.byref(c), 1, 1, None, None, None, 1, 1, 1, 1, 1, None, 256, big,
                      None)
    assert s == 1
    s = lib.moe_combine(ctypes.byref(c), 1, 1, 1, None, 1, None)
    assert s == 1
    # and the Expert Choice ones a top-k configuration
    tk = moe.make_config(synth.workload("switch_top1_cap"))
    s = lib.moe_route_expert_choice(ctypes.byref(tk), 1, 1, None, None, 1, 1, 1, 1, 1, 1, None,
                                    256, big, None)
    assert s == 1
    s = lib.moe_combine_expert_choice(ctypes.byref(tk), 1, 1, 1, None, 1, None)
    assert s == 1
    # missing slot table
    s = lib.moe_route_expert_choice(ctypes.byref(c), 1, 1, None, None, 1, 1, None, 1, 1, 1, None,
                                    256, big, None)
    assert s == 1


def test_expert_choice_workspace_holds_its_rows(lib):
    cfg = synth.workload("switch_expert_choice")
    T, d, F, E = cfg["T"], cfg["d_model"], cfg["d_ff"], cfg["E"]
    rows = E * moe.expert_capacity(cfg)
    # x_perm + H + Y for the E*C expert rows, plus the [E, T] logits and slot table
    assert moe.workspace_size(cfg) >= rows * (2 * d + F) * 2 + 2 * E * T * 4


def test_mx_unsupported_configurations_are_rejected(lib):
    """MX FP8 experts need a bf16 layer, top-k routing, no shared experts and
    d_model, d_ff multiples of 128: anything else is MOE_ERR_UNSUPPORTED on
    the host."""
    base = synth.workload("mixtral_top2", T=64, d_model=256, d_ff=512, experts="mxfp8")
    assert moe.workspace_size(base) > 0
    for bad in (dict(d_model=192), dict(d_ff=320), dict(n_shared=1), dict(dtype="f32"),
                dict(route="expert_choice", capacity_factor=1.0)):
        with pytest.raises(moe.MoEError) as ei:
            moe.workspace_size(dict(base, **bad))
        assert ei.value.status == 2, bad


def test_mxfp8_weight_bytes(lib):
    # codes, scale blocks, then 4 KB scale tile records per (expert, 128-K
    # stage, 256-row tile)
    assert moe.mxfp8_weight_bytes(8, 256, 128) == 8 * 256 * 128 * 33 // 32 + 8 * 1 * 1 * 4096
    assert moe.mxfp8_weight_bytes(2, 384, 256) == 2 * 384 * 256 * 33 // 32 + 2 * 2 * 2 * 4096
    for G, N, K in ((8, 200, 128), (8, 256, 96)):
        with pytest.raises(moe.MoEError) as ei:
            moe.mxfp8_weight_bytes(G, N, K)
        assert ei.value.status == 2
