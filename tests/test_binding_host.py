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


# ---- the wrappers' tensor checks (before any pointer reaches the C ABI)

def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def _raises(fn, match):
    with pytest.raises(ValueError, match=match):
        fn()


def test_attn_fwd_rejects_inconsistent_tensors():
    q, k, v = _t(1, 4, 64, 64), _t(1, 2, 96, 64), _t(1, 2, 96, 64)
    _raises(lambda: ga.attn_fwd(q.transpose(2, 3), k, v), "q must be contiguous")
    _raises(lambda: ga.attn_fwd(q, k, _t(1, 2, 80, 64)), r"v has shape \[1, 2, 80, 64\]")
    _raises(lambda: ga.attn_fwd(q, _t(1, 2, 96, 32), v), r"k has shape")
    _raises(lambda: ga.attn_fwd(q, _t(2, 2, 96, 64), _t(2, 2, 96, 64)), r"k has shape")
    _raises(lambda: ga.attn_fwd(q, k.float(), v), "k has dtype")
    _raises(lambda: ga.attn_fwd(q.half(), k.half(), v.half()), "q has dtype")
    _raises(lambda: ga.attn_fwd(q[0], k, v), "4-D")
    _raises(lambda: ga.attn_fwd(q, k, v, o=_t(1, 4, 64, 32)), r"o has shape")
    _raises(lambda: ga.attn_fwd(q, k, v, lse=_t(1, 4, 64, dtype=torch.bfloat16)), "lse has dtype")
    spec = ga.MaskSpec(kind=ga.CAUSAL, key_bias=_t(1, 4, 95, dtype=torch.float32))
    _raises(lambda: ga.attn_fwd(q, k, v, 0.0, spec), r"mask.key_bias has shape")
    # consistent shapes on the CPU: only the device check is left
    _raises(lambda: ga.attn_fwd(q, k, v), "must be on a CUDA device")


def test_attn_bwd_rejects_inconsistent_tensors():
    q, k, v = _t(1, 4, 64, 192), _t(1, 4, 64, 192), _t(1, 4, 64, 128)
    o, do, lse = _t(1, 4, 64, 128), _t(1, 4, 64, 128), _t(1, 4, 64, dtype=torch.float32)
    _raises(lambda: ga.attn_bwd(q, k, v, _t(1, 4, 64, 192), do, lse), r"o has shape")
    _raises(lambda: ga.attn_bwd(q, k, v, o, do.float(), lse), "dout has dtype")
    _raises(lambda: ga.attn_bwd(q, k, v, o, do, lse, dk=_t(1, 4, 64, 128)), r"dk has shape")
    _raises(lambda: ga.attn_bwd(q, k, v, o, do, lse, dkey_bias=_t(1, 4, 64)), "dkey_bias has dtype")
    _raises(lambda: ga.attn_bwd(q, k, v, o, do, lse), "must be on a CUDA device")


def test_splitkv_wrappers_reject_inconsistent_tensors():
    q, k, v = _t(2, 8, 1, 128), _t(2, 2, 256, 128), _t(2, 2, 256, 128)
    _raises(lambda: ga.attn_fwd_splitkv(q, k, _t(2, 2, 255, 128), num_splits=2), r"v has shape")
    _raises(lambda: ga.attn_fwd_splitkv(q, k, v, o=_t(2, 8, 1, 64)), r"o has shape")
    _raises(lambda: ga.attn_fwd_splitkv_noalloc(q, k, v, lse=_t(2, 8, 2, dtype=torch.float32)), r"lse has shape")
    kc, vc = _t(10, 2, 128, 128), _t(10, 2, 128, 128)
    pt, sl = _t(2, 5, dtype=torch.int32), _t(2, dtype=torch.int32)
    _raises(lambda: ga.attn_fwd_splitkv_paged(q, kc, vc, pt.long(), sl), "page_table has dtype")
    _raises(lambda: ga.attn_fwd_splitkv_paged(q, kc, vc, pt, _t(3, dtype=torch.int32)), r"seqlens_k has shape")
    _raises(lambda: ga.attn_fwd_splitkv_paged(q, _t(10, 2, 64, 128), vc, pt, sl), r"k_cache has shape")
    _raises(lambda: ga.attn_fwd_splitkv_paged(q, kc, vc, pt, sl), "must be on a CUDA device")
