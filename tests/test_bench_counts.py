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


def test_fsa_test_setup_fixture_drives_the_seeds_and_splits():
    """The [FSA] Testing section's set-up (tests/golden/fsa_pr148_test_setup.txt):
    split counts 1/2/4/8/16 and seed 42. The split-KV parity tests take their
    split counts from the fixture; the bench's decode workload and the seeded
    input generator's default must agree with it."""
    import inspect

    import bench
    from block_sparse_attention_tma_gb300 import synth
    from conftest import golden_setup

    g = golden_setup()
    assert g["splits"] == [1, 2, 4, 8, 16]
    assert tuple(g["splits"]) == bench.DECODE["splits"]
    assert inspect.signature(synth.make_inputs).parameters["seed"].default == g["seed"]
    assert inspect.signature(synth.make_device_inputs).parameters["seed"].default == g["seed"]
    # the head dims the bf16 tensor-core path supports are among the page's
    assert {32, 64, 128, 192} <= set(g["head_dims"])
