"""The CTA-pair (tcgen05 cta_group::2) dK/dV kernel against the oracle.

"Enable 2CTA for SM100 block-sparse backward" (Summary): the backward's kv
sub-tiling of a sparse block lets two CTAs share each MMA (M = 256 keys). The
kernel is selected with gbattn_set_dkdv_cta_pair(1); every case here also
runs the one-CTA kernel on the same inputs. Both must match the oracle at the
backward tolerance (max |err| / max |ref| <= 5e-2), the pair kernel must be
bitwise reproducible, and dQ (the same query-parallel kernel either way) must
be identical. Cases: the MLA head dims 192 / 128 and 128 / 128, ragged and
unequal lengths, an odd number of key tiles (the last pair's second CTA has
no keys), sparse tiles of 256 and 512 keys and no lists, grouped-query heads,
softcap, a key bias with its gradient, and the dynamic mask walked with keep
bits.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga
from helpers import Case, assert_no_device_error, check_dbias, check_grad, f64

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Sq, Sk, Dqk, Dv, kind, extras
    (1, 2, 700, 700, 192, 128, "causal", dict(slope=0.01)),
    (1, 2, 513, 900, 128, 128, "sliding", dict(window=200, sparse=(256, 256))),
    (2, 2, 384, 384, 192, 128, "none", dict(lists=False, sparse=None)),
    (1, 4, 300, 640, 192, 128, "prefix_lm", dict(prefix_len=100, Hkv=2)),
    (1, 2, 1000, 1000, 128, 128, "block_diag", dict(block_size=256, sparse=(256, 256))),
    (1, 1, 400, 400, 128, 128, "causal", dict(softcap=30.0, sparse=(128, 256))),
    (1, 1, 900, 900, 192, 128, "dynamic", dict(topk=300, gather=False, sparse=(128, 256))),
    (1, 2, 260, 1300, 192, 128, "causal", dict(sparse=(256, 512))),
]


def _bwd(c, o, lse, mode, dbias=False):
    prev = ga.set_dkdv_cta_pair(mode)
    try:
        db = c.dbias_buffer() if dbias else None
        dq, dk, dv = c.bwd(o, lse, dkey_bias=db)
        torch.cuda.synchronize()
    finally:
        ga.set_dkdv_cta_pair(prev)
    return dq, dk, dv, db


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[6]}-{c[2]}x{c[3]}-d{c[4]}")
def test_pair_dkdv_matches_oracle_and_one_cta_kernel(case):
    B, H, Sq, Sk, Dqk, Dv, kind, ex = case
    c = Case(B, H, Sq, Sk, Dqk, Dv, kind, **ex)
    o, lse = c.fwd()
    one = _bwd(c, o, lse, 0)
    pair = _bwd(c, o, lse, 1)
    again = _bwd(c, o, lse, 1)
    assert_no_device_error()
    for x, y in zip(pair[:3], again[:3]):
        assert torch.equal(x, y), "pair kernel not bitwise reproducible"
    assert torch.equal(one[0], pair[0]), "dQ differs"
    G = c.G
    for b in range(B):
        for h in range(H):
            dq_r, dk_r, dv_r, _ = c.problem(b, h).backward(c.h["do"][b, h])
            check_grad(f64(pair[0][b, h]), dq_r, "dQ")
            if h % G == 0:  # dK / dV of key/value head h // G: the sum over its query heads
                dk_sum = sum(c.problem(b, h + g).backward(c.h["do"][b, h + g])[1] for g in range(G))
                dv_sum = sum(c.problem(b, h + g).backward(c.h["do"][b, h + g])[2] for g in range(G))
                for name, grads in (("one-CTA", one), ("pair", pair)):
                    check_grad(f64(grads[1][b, h // G]), dk_sum, f"dK ({name})")
                    check_grad(f64(grads[2][b, h // G]), dv_sum, f"dV ({name})")


def test_pair_dkdv_key_bias_gradient():
    c = Case(1, 2, 640, 700, 192, 128, "causal", use_bias=True, slope=0.01)
    o, lse = c.fwd()
    dq, dk, dv, db = _bwd(c, o, lse, 1, dbias=True)
    assert_no_device_error()
    for h in range(2):
        p = c.problem(0, h)
        dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, h])
        check_grad(f64(dk[0, h]), dk_r, "dK")
        check_grad(f64(dv[0, h]), dv_r, "dV")
        check_dbias(f64(db[0, h]), p.dkey_bias(c.h["do"][0, h]))


