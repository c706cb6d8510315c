"""CPU oracle for the sparse-MoE FFN forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product package never does.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (OracleConfig, moe_forward, router_logits, softmax,  # noqa: F401
                         select_topk, gate, capacity, dispatch, gelu,
                         expert_ffn, load_balance, router_z_loss)
