"""bench.py's FLOP convention counts the allowed (q, k) pairs of each mask in
closed form; these CPU tests check those counts against the oracle's element
mask summed pair by pair, and the dynamic workload's count (kept key p seen by
rows p .. S-1) against the oracle's keep set."""
import numpy as np
import pytest
import torch

import bench
from oracle import attention as orc


@pytest.mark.parametrize("S", [1, 7, 300, 1031])
@pytest.mark.parametrize("kind,kw", [("causal", {}), ("sliding", dict(window_left=100)),
                                     ("sliding", dict(window_left=5000)), ("block_diag", dict(block_size=64)),
                                     ("block_diag", dict(block_size=4096)), ("prefix_lm", dict(prefix_len=37)),
                                     ("prefix_lm", dict(prefix_len=5000))])
def test_mask_pairs_match_oracle(S, kind, kw):
    code = {"causal": orc.CAUSAL, "sliding": orc.SLIDING, "block_diag": orc.BLOCK_DIAG,
            "prefix_lm": orc.PREFIX_LM}[kind]
    m = orc.allowed(code, S, S, np.arange(S), np.arange(S), **kw)
    assert bench.mask_pairs(kind, S, **kw) == int(m.sum())


def test_dynamic_pair_count_matches_oracle():
    S, topk = 700, 150
    bias = torch.randn(S, generator=torch.Generator().manual_seed(3))
    kept = torch.topk(bias.double(), topk).indices
    count = int((S - kept).sum())
    keep = orc.topk_keep(bias.double().numpy(), topk)
    m = orc.allowed(orc.DYNAMIC_TOPK, S, S, np.arange(S), np.arange(S), keep=keep)
    assert count == int(m.sum())
