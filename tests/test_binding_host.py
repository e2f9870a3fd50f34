"""Host-side helpers of the binding that run without a GPU: the TABLE mask
packer's bit order (bit j % 32 of word j // 32 of row i = pair (i, j)),
checked against a brute-force packer, at widths around the 32-key word
boundary and with bit 31 (the int32 sign bit) set."""
import numpy as np
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga


def _brute(mask):
    *lead, sq, sk = mask.shape
    nw = (sk + 31) // 32
    out = np.zeros((*lead, sq, nw), dtype=np.uint32)
    it = np.ndindex(*mask.shape)
    for idx in it:
        if mask[idx]:
            *pre, i, j = idx
            out[(*pre, i, j // 32)] |= np.uint32(1) << np.uint32(j % 32)
    return out.view(np.int32)


@pytest.mark.parametrize("sk", [1, 31, 32, 33, 64, 100])
def test_pack_mask_table_bit_order(sk):
    rng = np.random.default_rng(sk)
    m = rng.random((3, sk)) < 0.5
    m[0, :] = True  # every bit of the row, incl. bit 31 of full words
    got = ga.pack_mask_table(torch.from_numpy(m)).numpy()
    assert got.dtype == np.int32 and got.shape == (3, (sk + 31) // 32)
    assert np.array_equal(got, _brute(m))


def test_pack_mask_table_per_head_layout():
    rng = np.random.default_rng(7)
    m = rng.random((2, 3, 5, 70)) < 0.3
    got = ga.pack_mask_table(torch.from_numpy(m)).numpy()
    assert got.shape == (2, 3, 5, 3)
    assert np.array_equal(got, _brute(m))
