"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; torch supplies device
memory and the current stream.  Calls raise ``MoEError`` on any non-OK status,
and loading fails loudly when ``libmoe.so`` has not been built.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

ROUTES = {"softmax_topk": 0, "topk_softmax": 1, "biased_softmax": 2, "expert_choice": 3}
DTYPES = {"f32": 0, "bf16": 1}
AUX_F = {"topk_count": 0, "argmax": 1}
ACTS = {"gelu": 0, "silu": 1, "swiglu": 2}
EXPERT_FMTS = {"dense": 0, "mxfp8": 1}
TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        self.fn = fn
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


class Config(ctypes.Structure):
    """moe_config of include/moe.h (field order and types must match)."""
    _fields_ = [
        ("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
        ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
        ("capacity_factor", ctypes.c_float), ("min_capacity", ctypes.c_int32),
        ("route", ctypes.c_int32), ("renorm", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("has_bias", ctypes.c_int32), ("aux_alpha", ctypes.c_float), ("aux_f", ctypes.c_int32),
        ("act", ctypes.c_int32), ("y_f32", ctypes.c_int32), ("expert_fmt", ctypes.c_int32),
    ]


def make_config(cfg: dict) -> Config:
    """Config from a workload dict (keys as in ``synth.WORKLOADS``)."""
    c = Config()
    c.T, c.d_model, c.d_ff = int(cfg["T"]), int(cfg["d_model"]), int(cfg["d_ff"])
    c.E, c.k, c.n_shared = int(cfg["E"]), int(cfg["k"]), int(cfg.get("n_shared", 0))
    c.capacity_factor = float(cfg.get("capacity_factor", 0.0))
    c.min_capacity = int(cfg.get("min_capacity", 0))
    r = cfg.get("route", "softmax_topk")
    c.route = ROUTES[r] if isinstance(r, str) else int(r)
    c.renorm = int(cfg.get("renorm", 1))
    dt = cfg.get("dtype", "bf16")
    c.dtype = DTYPES[dt] if isinstance(dt, str) else int(dt)
    c.has_bias = int(cfg.get("has_bias", 0))
    c.aux_alpha = float(cfg.get("aux_alpha", 0.01))
    af = cfg.get("aux_f", "topk_count")
    c.aux_f = AUX_F[af] if isinstance(af, str) else int(af)
    a = cfg.get("act", "gelu")
    c.act = ACTS[a] if isinstance(a, str) else int(a)
    c.y_f32 = int(cfg.get("y_f32", 0))
    f = cfg.get("experts", "dense")
    c.expert_fmt = EXPERT_FMTS[f] if isinstance(f, str) else int(f)
    return c


def mx_experts(cfg: dict) -> bool:
    """True when the expert weights are packed MX FP8 buffers."""
    return cfg.get("experts", "dense") in ("mxfp8", EXPERT_FMTS["mxfp8"])


def y_dtype(cfg: dict) -> torch.dtype:
    """Element type of the expert outputs y_perm / y_shared: the layer dtype,
    or fp32 when the configuration keeps them so (``y_f32``)."""
    return torch.float32 if cfg.get("y_f32", 0) else TORCH_DTYPES[cfg["dtype"]]


def w1_rows(cfg: dict) -> int:
    """Rows of each expert's first weight: 2 d_ff for SwiGLU (the gate
    projection's rows, then the up projection's), else d_ff."""
    return 2 * cfg["d_ff"] if cfg.get("act", "gelu") in ("swiglu", ACTS["swiglu"]) else cfg["d_ff"]


_lib = None
_P = ctypes.c_void_p
_CFG = ctypes.POINTER(Config)
_SIGNATURES = {
    "moe_workspace_size": [_CFG, ctypes.POINTER(ctypes.c_size_t)],
    "moe_workspace_init": [_P, ctypes.c_size_t, _P],
    "moe_route": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_permute": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_permute_noalloc": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_grouped_ffn": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                        ctypes.c_size_t, _P],
    "moe_combine": [_CFG, _P, _P, _P, _P, _P, _P],
    "moe_forward": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                    _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_check_status": [_P, _P],
    "moe_expert_capacity": [_CFG, ctypes.POINTER(ctypes.c_int32)],
    "moe_route_expert_choice": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                ctypes.c_size_t, _P],
    "moe_permute_expert_choice": [_CFG, _P, _P, _P, _P, _P],
    "moe_combine_expert_choice": [_CFG, _P, _P, _P, _P, _P, _P],
    "moe_mxfp8_weight_bytes": [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                               ctypes.POINTER(ctypes.c_size_t)],
    "moe_quantize_mxfp8": [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                           _P, _P],
}


def lib() -> ctypes.CDLL:
    """The loaded libmoe (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoEError("load libmoe.so", -1) from FileNotFoundError(
                f"{LIB_PATH} missing: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().moe_status_string(int(s)).decode()


def _call(name: str, *args) -> None:
    s = getattr(lib(), name)(*args)
    if s != 0:
        raise MoEError(name, s)


def _p(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _want(t: Optional[torch.Tensor], name: str, shape, dtype, allow_none=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


# ------------------------------------------------------------------ MX FP8 weights
def mxfp8_weight_bytes(G: int, N: int, K: int) -> int:
    n = ctypes.c_size_t(0)
    _call("moe_mxfp8_weight_bytes", int(G), int(N), int(K), ctypes.byref(n))
    return int(n.value)


def quantize_mxfp8(w: torch.Tensor, glu: bool = False, stream=None) -> torch.Tensor:
    """moe_quantize_mxfp8: packs bf16 expert weights [G, N, K] into one uint8
    buffer (e4m3 codes, then the scale blocks); glu interleaves the gate and up
    halves of a SwiGLU w1 in 64-row halves."""
    if w.dim() != 3 or w.dtype != torch.bfloat16 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("w must be a contiguous [G, N, K] bf16 CUDA tensor")
    G, N, K = w.shape
    out = torch.empty(mxfp8_weight_bytes(G, N, K), dtype=torch.uint8, device=w.device)
    _call("moe_quantize_mxfp8", _p(w), int(G), int(N), int(K), int(bool(glu)), _p(out),
          _stream(stream))
    return out


def _want_weights(cfg, w1, w2, dt):
    """Expert weights: [E, F1, d] and [E, d, F] in dtype, or their packed MX
    FP8 buffers."""
    d, F, E = cfg["d_model"], cfg["d_ff"], cfg["E"]
    F1 = w1_rows(cfg)
    if mx_experts(cfg):
        _want(w1, "w1", (mxfp8_weight_bytes(E, F1, d),), torch.uint8)
        _want(w2, "w2", (mxfp8_weight_bytes(E, d, F),), torch.uint8)
    else:
        _want(w1, "w1", (E, F1, d), dt)
        _want(w2, "w2", (E, d, F), dt)


# ------------------------------------------------------------------ workspace
def workspace_size(cfg: dict) -> int:
    n = ctypes.c_size_t(0)
    _call("moe_workspace_size", ctypes.byref(make_config(cfg)), ctypes.byref(n))
    return int(n.value)


def new_workspace(cfg: dict, device="cuda", stream=None) -> torch.Tensor:
    """Allocates (through torch) and initialises a workspace for ``cfg``."""
    n = workspace_size(cfg)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _call("moe_workspace_init", _p(ws), ws.numel(), _stream(stream))
    return ws


def check_status(ws: torch.Tensor, stream=None) -> None:
    _call("moe_check_status", _p(ws), _stream(stream))


def expert_choice(cfg: dict) -> bool:
    return cfg.get("route") in ("expert_choice", ROUTES["expert_choice"])


def expert_capacity(cfg: dict) -> int:
    """C of the configuration (tokens per expert under Expert Choice), or -1
    for top-k routing without a capacity limit."""
    c = ctypes.c_int32(0)
    _call("moe_expert_capacity", ctypes.byref(make_config(cfg)), ctypes.byref(c))
    return int(c.value)


def routed_rows(cfg: dict) -> int:
    """Expert-ordered rows of x_perm / y_perm: T*k, or E*C under Expert Choice."""
    return cfg["E"] * expert_capacity(cfg) if expert_choice(cfg) else cfg["T"] * cfg["k"]


# ------------------------------------------------------------------ steps
def route(cfg, x, w_g, topk_idx, topk_w, f, P, aux, ws, logit_bias=None, select_bias=None,
          logits=None, z_loss=None, stream=None):
    T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(x, "x", (T, d), dt)
    _want(w_g, "w_g", (d, E), dt)
    _want(topk_idx, "topk_idx", (T, k), torch.int32)
    _want(topk_w, "topk_w", (T, k), torch.float32)
    _want(f, "f", (E,), torch.float32)
    _want(P, "P", (E,), torch.float32)
    _want(aux, "aux", (1,), torch.float32)
    _want(logit_bias, "logit_bias", (E,), torch.float32, allow_none=True)
    _want(select_bias, "select_bias", (E,), torch.float32, allow_none=True)
    _want(logits, "logits", (T, E), torch.float32, allow_none=True)
    _want(z_loss, "z_loss", (1,), torch.float32, allow_none=True)
    _call("moe_route", ctypes.byref(make_config(cfg)), _p(x), _p(w_g), _p(logit_bias),
          _p(select_bias), _p(logits), _p(topk_idx), _p(topk_w), _p(f), _p(P), _p(aux),
          _p(z_loss), _p(ws), ws.numel(), _stream(stream))


def permute(cfg, x, topk_idx, counts, kept, offsets, perm_token, slot_of, x_perm, ws,
            stream=None):
    T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(x, "x", (T, d), dt)
    _want(topk_idx, "topk_idx", (T, k), torch.int32)
    _want(counts, "counts", (E,), torch.int32)
    _want(kept, "kept", (E,), torch.int32)
    _want(offsets, "offsets", (E + 1,), torch.int32)
    _want(perm_token, "perm_token", (T * k,), torch.int32)
    _want(slot_of, "slot_of", (T * k,), torch.int32)
    _want(x_perm, "x_perm", (T * k, d), dt)
    _call("moe_permute", ctypes.byref(make_config(cfg)), _p(x), _p(topk_idx), _p(counts),
          _p(kept), _p(offsets), _p(perm_token), _p(slot_of), _p(x_perm), _p(ws), ws.numel(),
          _stream(stream))


# limits of moe_permute_noalloc (MOE_PERMUTE_NOALLOC_MAX_* in moe.h): T*k, and
# the per-chunk expert counts 32*ceil(ceil(T/32)/32)*E (each expert's row of
# 32-token chunk counts padded to a multiple of 32 chunks)
PERMUTE_NOALLOC_MAX_ASSIGNMENTS = 1 << 20
PERMUTE_NOALLOC_MAX_CHUNK_COUNTS = 1 << 20


def permute_noalloc(cfg, x, topk_idx, counts, kept, offsets, perm_token, slot_of, x_perm,
                    stream=None):
    """moe_permute_noalloc: the dispatch of ``permute`` without a workspace.

    For callers that cannot allocate device memory themselves: its scratch is a
    fixed 8 MiB array inside the library.  The first call on a device must come
    before any stream capture; calls that may overlap on the GPU race, because
    they share that array.  Raises MoEError (MOE_ERR_UNSUPPORTED) when
    T*k > PERMUTE_NOALLOC_MAX_ASSIGNMENTS or 32*ceil(ceil(T/32)/32)*E >
    PERMUTE_NOALLOC_MAX_CHUNK_COUNTS.
    """
    T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(x, "x", (T, d), dt)
    _want(topk_idx, "topk_idx", (T, k), torch.int32)
    _want(counts, "counts", (E,), torch.int32)
    _want(kept, "kept", (E,), torch.int32)
    _want(offsets, "offsets", (E + 1,), torch.int32)
    _want(perm_token, "perm_token", (T * k,), torch.int32)
    _want(slot_of, "slot_of", (T * k,), torch.int32)
    _want(x_perm, "x_perm", (T * k, d), dt)
    _call("moe_permute_noalloc", ctypes.byref(make_config(cfg)), _p(x), _p(topk_idx),
          _p(counts), _p(kept), _p(offsets), _p(perm_token), _p(slot_of), _p(x_perm),
          _stream(stream))


def grouped_ffn(cfg, x_perm, offsets, w1, w2, y_perm, ws, b1=None, b2=None, x=None, ws1=None,
                wsb1=None, ws2=None, wsb2=None, y_shared=None, stream=None):
    T, d, F, E, k, S = (cfg["T"], cfg["d_model"], cfg["d_ff"], cfg["E"], cfg["k"],
                        cfg.get("n_shared", 0))
    dt = TORCH_DTYPES[cfg["dtype"]]
    F1 = w1_rows(cfg)
    R = routed_rows(cfg)
    _want(x_perm, "x_perm", (R, d), dt)
    _want(offsets, "offsets", (E + 1,), torch.int32)
    _want_weights(cfg, w1, w2, dt)
    _want(b1, "b1", (E, F1), dt, allow_none=not cfg.get("has_bias", 0))
    _want(b2, "b2", (E, d), dt, allow_none=not cfg.get("has_bias", 0))
    _want(y_perm, "y_perm", (R, d), y_dtype(cfg))
    if S:
        _want(x, "x", (T, d), dt)
        _want(ws1, "ws1", (S, F1, d), dt)
        _want(wsb1, "wsb1", (S, F1), dt, allow_none=True)
        _want(ws2, "ws2", (S, d, F), dt)
        _want(y_shared, "y_shared", (S, T, d), y_dtype(cfg))
    _call("moe_grouped_ffn", ctypes.byref(make_config(cfg)), _p(x_perm), _p(offsets), _p(w1),
          _p(b1), _p(w2), _p(b2), _p(x), _p(ws1), _p(wsb1), _p(ws2), _p(wsb2), _p(y_perm),
          _p(y_shared), _p(ws), ws.numel(), _stream(stream))


def route_expert_choice(cfg, x, w_g, ec_token, ec_w, ec_slot, f, P, aux, ws, logit_bias=None,
                        logits=None, z_loss=None, stream=None):
    T, d, E = cfg["T"], cfg["d_model"], cfg["E"]
    C = expert_capacity(cfg)
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(x, "x", (T, d), dt)
    _want(w_g, "w_g", (d, E), dt)
    _want(ec_token, "ec_token", (E, C), torch.int32)
    _want(ec_w, "ec_w", (E, C), torch.float32)
    _want(ec_slot, "ec_slot", (E, T), torch.int32)
    for n, t in (("f", f), ("P", P)):
        _want(t, n, (E,), torch.float32)
    _want(aux, "aux", (1,), torch.float32)
    _want(logit_bias, "logit_bias", (E,), torch.float32, allow_none=True)
    _want(logits, "logits", (T, E), torch.float32, allow_none=True)
    _want(z_loss, "z_loss", (1,), torch.float32, allow_none=True)
    _call("moe_route_expert_choice", ctypes.byref(make_config(cfg)), _p(x), _p(w_g),
          _p(logit_bias), _p(logits), _p(ec_token), _p(ec_w), _p(ec_slot), _p(f), _p(P),
          _p(aux), _p(z_loss), _p(ws), ws.numel(), _stream(stream))


def permute_expert_choice(cfg, x, ec_token, offsets, x_perm, stream=None):
    T, d, E = cfg["T"], cfg["d_model"], cfg["E"]
    C = expert_capacity(cfg)
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(x, "x", (T, d), dt)
    _want(ec_token, "ec_token", (E, C), torch.int32)
    _want(offsets, "offsets", (E + 1,), torch.int32)
    _want(x_perm, "x_perm", (E * C, d), dt)
    _call("moe_permute_expert_choice", ctypes.byref(make_config(cfg)), _p(x), _p(ec_token),
          _p(offsets), _p(x_perm), _stream(stream))


def combine_expert_choice(cfg, y_perm, ec_slot, ec_w, out, y_shared=None, stream=None):
    T, d, E, S = cfg["T"], cfg["d_model"], cfg["E"], cfg.get("n_shared", 0)
    C = expert_capacity(cfg)
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(y_perm, "y_perm", (E * C, d), y_dtype(cfg))
    _want(ec_slot, "ec_slot", (E, T), torch.int32)
    _want(ec_w, "ec_w", (E, C), torch.float32)
    _want(out, "out", (T, d), dt)
    if S:
        _want(y_shared, "y_shared", (S, T, d), y_dtype(cfg))
    _call("moe_combine_expert_choice", ctypes.byref(make_config(cfg)), _p(y_perm), _p(ec_slot),
          _p(ec_w), _p(y_shared), _p(out), _stream(stream))


def combine(cfg, y_perm, slot_of, topk_w, out, y_shared=None, stream=None):
    T, d, k, S = cfg["T"], cfg["d_model"], cfg["k"], cfg.get("n_shared", 0)
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(y_perm, "y_perm", (T * k, d), y_dtype(cfg))
    _want(slot_of, "slot_of", (T * k,), torch.int32)
    _want(topk_w, "topk_w", (T, k), torch.float32)
    _want(out, "out", (T, d), dt)
    if S:
        _want(y_shared, "y_shared", (S, T, d), y_dtype(cfg))
    _call("moe_combine", ctypes.byref(make_config(cfg)), _p(y_perm), _p(slot_of), _p(topk_w),
          _p(y_shared), _p(out), _stream(stream))


def forward(cfg, x, w_g, w1, w2, out, ws, b1=None, b2=None, ws1=None, wsb1=None, ws2=None,
            wsb2=None, logit_bias=None, select_bias=None, topk_idx=None, topk_w=None,
            counts=None, f=None, P=None, aux=None, z_loss=None, stream=None):
    """The whole layer in one call (route -> permute -> grouped FFN -> combine)."""
    T, d, F, E, k, S = (cfg["T"], cfg["d_model"], cfg["d_ff"], cfg["E"], cfg["k"],
                        cfg.get("n_shared", 0))
    dt = TORCH_DTYPES[cfg["dtype"]]
    _want(x, "x", (T, d), dt)
    _want(w_g, "w_g", (d, E), dt)
    F1 = w1_rows(cfg)
    _want_weights(cfg, w1, w2, dt)
    _want(b1, "b1", (E, F1), dt, allow_none=True)
    _want(out, "out", (T, d), dt)
    # under Expert Choice topk_idx / topk_w carry the [E, C] taken tokens and weights
    sel = (E, expert_capacity(cfg)) if expert_choice(cfg) else (T, k)
    _want(topk_idx, "topk_idx", sel, torch.int32, allow_none=True)
    _want(topk_w, "topk_w", sel, torch.float32, allow_none=True)
    _want(counts, "counts", (E,), torch.int32, allow_none=True)
    for n, t in (("f", f), ("P", P)):
        _want(t, n, (E,), torch.float32, allow_none=True)
    _want(aux, "aux", (1,), torch.float32, allow_none=True)
    _want(z_loss, "z_loss", (1,), torch.float32, allow_none=True)
    if S:
        _want(ws1, "ws1", (S, F1, d), dt)
        _want(wsb1, "wsb1", (S, F1), dt, allow_none=True)
        _want(ws2, "ws2", (S, d, F), dt)
    _call("moe_forward", ctypes.byref(make_config(cfg)), _p(x), _p(w_g), _p(logit_bias),
          _p(select_bias), _p(w1), _p(b1), _p(w2), _p(b2), _p(ws1), _p(wsb1), _p(ws2),
          _p(wsb2), _p(out), _p(topk_idx), _p(topk_w), _p(counts), _p(f), _p(P), _p(aux),
          _p(z_loss), _p(ws), ws.numel(), _stream(stream))


class MoELayer:
    """One MoE FFN layer whose weights stay resident on the device.

    ``inputs`` holds the weight tensors named as in ``synth.make_inputs``
    (x is ignored).  ``__call__(x)`` runs ``moe_forward`` and returns the
    output plus the routing statistics, all as device tensors.
    """

    def __init__(self, cfg: dict, inputs: dict, device="cuda"):
        self.cfg = dict(cfg)
        self.w = {k: v for k, v in inputs.items() if k != "x"}
        self.device = torch.device(device)
        if mx_experts(cfg) and self.w["w1"].dtype != torch.uint8:
            # MX FP8 experts: pack the bf16 weights once (on the device)
            glu = cfg.get("act", "gelu") in ("swiglu", ACTS["swiglu"])
            self.w["w1"] = quantize_mxfp8(self.w["w1"], glu=glu)
            self.w["w2"] = quantize_mxfp8(self.w["w2"])
        self.ws = new_workspace(self.cfg, self.device)
        T, d, E, k = cfg["T"], cfg["d_model"], cfg["E"], cfg["k"]
        dt = TORCH_DTYPES[cfg["dtype"]]
        self.out = torch.empty((T, d), dtype=dt, device=self.device)
        # Expert Choice: the [E, C] taken tokens and their weights instead
        sel = (E, expert_capacity(cfg)) if expert_choice(cfg) else (T, k)
        self.topk_idx = torch.empty(sel, dtype=torch.int32, device=self.device)
        self.topk_w = torch.empty(sel, dtype=torch.float32, device=self.device)
        self.counts = torch.empty((E,), dtype=torch.int32, device=self.device)
        self.f = torch.empty((E,), dtype=torch.float32, device=self.device)
        self.P = torch.empty((E,), dtype=torch.float32, device=self.device)
        self.aux = torch.empty((1,), dtype=torch.float32, device=self.device)
        self.z_loss = torch.empty((1,), dtype=torch.float32, device=self.device)

    def __call__(self, x: torch.Tensor, stream=None) -> dict:
        w = self.w
        forward(self.cfg, x, w["w_g"], w["w1"], w["w2"], self.out, self.ws, b1=w.get("b1"),
                b2=w.get("b2"), ws1=w.get("ws1"), wsb1=w.get("wsb1"), ws2=w.get("ws2"),
                wsb2=w.get("wsb2"), logit_bias=w.get("logit_bias"),
                select_bias=w.get("select_bias"), topk_idx=self.topk_idx, topk_w=self.topk_w,
                counts=self.counts, f=self.f, P=self.P, aux=self.aux, z_loss=self.z_loss,
                stream=stream)
        return self._outputs()

    def _outputs(self) -> dict:
        return dict(out=self.out, topk_idx=self.topk_idx, topk_w=self.topk_w,
                    counts=self.counts, f=self.f, P=self.P, aux=self.aux, z_loss=self.z_loss)


class GraphedMoELayer(MoELayer):
    """MoELayer whose forward is captured once in a CUDA graph.

    ``__call__(x)`` copies x into the graph's static input buffer (stream
    ordered, so a pinned host tensor is copied asynchronously) and replays the
    captured moe_forward: one graph launch per layer call instead of one
    ctypes call plus ~9 kernel launches.  The weights and outputs are the
    same device tensors as the eager layer's.
    """

    def __init__(self, cfg: dict, inputs: dict, device="cuda"):
        super().__init__(cfg, inputs, device)
        T, d = cfg["T"], cfg["d_model"]
        self.x_static = torch.zeros((T, d), dtype=TORCH_DTYPES[cfg["dtype"]], device=self.device)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):          # warm-up: kernel attributes, tensor-map encoder
            MoELayer.__call__(self, self.x_static)
        torch.cuda.current_stream(self.device).wait_stream(side)
        torch.cuda.synchronize(self.device)
        check_status(self.ws)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            MoELayer.__call__(self, self.x_static)

    def __call__(self, x: Optional[torch.Tensor] = None, stream=None) -> dict:
        if x is not None:
            self.x_static.copy_(x, non_blocking=True)
        self.graph.replay()
        return self._outputs()


class StreamedMoELayer:
    """Layer calls on pinned host tensors with the copies overlapped.

    ``submit(x_host, out_host)`` enqueues one call: the host-to-device copy of
    x, the graphed moe_forward and the device-to-host copy of the output (and
    of aux into ``aux_host`` when given), each on its own CUDA stream, ordered
    by events.  Two graphed layers take turns, so the input copy of call i+1
    and the output copy of call i-1 run while call i computes, and no call
    overwrites a buffer that a copy of an earlier call still reads.
    ``synchronize()`` waits for every submitted call; ``out_host`` of a call is
    complete after that (or after ``done_event(i)`` has fired).
    """

    def __init__(self, cfg: dict, inputs: dict, device="cuda"):
        self.device = torch.device(device)
        self.layers = [GraphedMoELayer(cfg, inputs, device) for _ in range(2)]
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(self.device) for _ in range(3))
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_in, self.ev_comp, self.ev_out = ev(), ev(), ev()
        self.calls = 0

    def submit(self, x_host: torch.Tensor, out_host: torch.Tensor,
               aux_host: Optional[torch.Tensor] = None) -> None:
        b = self.calls % 2
        L = self.layers[b]
        # x_static[b] is free once call - 2 has computed
        self.s_in.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_in):
            L.x_static.copy_(x_host, non_blocking=True)
            self.ev_in[b].record(self.s_in)
        # out[b] is free once the output copy of call - 2 has finished
        self.s_comp.wait_event(self.ev_in[b])
        self.s_comp.wait_event(self.ev_out[b])
        with torch.cuda.stream(self.s_comp):
            L.graph.replay()
            self.ev_comp[b].record(self.s_comp)
        self.s_out.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_out):
            out_host.copy_(L.out, non_blocking=True)
            if aux_host is not None:
                aux_host.copy_(L.aux, non_blocking=True)
            self.ev_out[b].record(self.s_out)
        self.calls += 1

    def done_event(self, i: int) -> torch.cuda.Event:
        """Event of the output copy of the last call submitted on call i's turn."""
        return self.ev_out[i % 2]

    def synchronize(self) -> None:
        self.s_out.synchronize()
        self.s_comp.synchronize()
        self.s_in.synchronize()
        for L in self.layers:
            check_status(L.ws)
