"""The acceptance rules of the oracle comparison on hand-made routings (no GPU).

A token whose k-th and (k+1)-th selection scores lie within the near-tie
margin may be routed differently by a device that sums in another order; its
device choice is accepted only when it is still a top-k set up to that margin.
These cases plant device choices on the CPU and check which ones pass."""

import numpy as np
import pytest
import torch

from oracle import compare
from sparse_mixture_experts_52_b300 import synth


def _case():
    """Four tokens, x_t = e_t, so token t's logits are row t of W_g.  Token 0
    has a near tie between experts 0 and 1 (2e-6 apart); the others are far
    from any tie."""
    cfg = synth.workload("tiny_fp32_top2", T=4, d_model=8, d_ff=8, E=8, k=2,
                         route="topk_softmax")
    inp = synth.make_inputs(cfg, device="cpu")
    x = torch.zeros(4, 8)
    x[torch.arange(4), torch.arange(4)] = 1.0
    wg = torch.zeros(8, 8)
    wg[0] = torch.tensor([3.0, 3.0 - 2e-6, 1.0, 0.5, 0.2, 0.1, 0.0, -1.0])
    wg[1] = torch.arange(8.0)
    wg[2] = -torch.arange(8.0)
    wg[3] = torch.tensor([0.0, 5.0, 1.0, 4.0, 2.0, 3.0, 0.5, 0.25])
    inp["x"], inp["w_g"] = x, wg
    return cfg, inp


def _oracle_idx(cfg, inp):
    return compare.run_oracle(cfg, inp, rows=[0]).gate.idx.astype(np.int32)


def test_oracle_order_passes_and_token_zero_is_a_near_tie():
    cfg, inp = _case()
    idx = _oracle_idx(cfg, inp)
    assert idx[0].tolist() == [0, 1]
    rep = compare.check_layer(cfg, inp, {"topk_idx": idx})
    assert rep.near_tie == [0] and rep.overridden == []


def test_swapped_near_tie_is_accepted_and_reported():
    cfg, inp = _case()
    idx = _oracle_idx(cfg, inp)
    idx[0] = [1, 0]
    rep = compare.check_layer(cfg, inp, {"topk_idx": idx})
    assert rep.overridden == [0]


@pytest.mark.parametrize("bad", [[0, 2], [2, 1], [0, 0], [0, 8]])
def test_near_tie_token_sent_elsewhere_fails(bad):
    """An expert outside the top-2 up to the margin (2, far below), a repeated
    expert, or one outside [0, E) is not a valid choice for a near-tie token."""
    cfg, inp = _case()
    idx = _oracle_idx(cfg, inp)
    idx[0] = bad
    with pytest.raises(AssertionError):
        compare.check_layer(cfg, inp, {"topk_idx": idx})


def test_token_without_tie_must_match_exactly():
    cfg, inp = _case()
    idx = _oracle_idx(cfg, inp)
    idx[1] = idx[1][::-1]
    with pytest.raises(AssertionError):
        compare.check_layer(cfg, inp, {"topk_idx": idx})
