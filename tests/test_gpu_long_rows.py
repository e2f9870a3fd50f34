"""Rows that visit more than 1024 key tiles, and a key tile visited by more
than 1024 query tiles. A CTA compacts the tiles it visits into a list in
shared memory that holds 1024 entries; past that every role of the CTA walks
the slots itself (the dense walk without lists, the list walk with them).
The forward and dQ kernels take that path for one 128-row query tile over
132,608 keys (1036 key tiles; dense, with lists, and over the compact tiles
of a dynamic top-k), the dK/dV kernel and its CTA-pair version for key tiles
under 132,608 query rows. Each case is checked against the fp64 oracle at the
parity tolerances.
"""
import pytest

import block_sparse_attention_tma_gb300 as ga
from helpers import Case, assert_no_device_error, check_grad, check_lse, check_out, f64

pytestmark = pytest.mark.gpu

LONG = 1036 * 128  # 132,608: 1036 tiles of 128, past the 1024-entry list


@pytest.mark.parametrize("kind,lists", [("none", False), ("causal", True)])
def test_query_tile_over_more_than_1024_key_tiles(kind, lists):
    # causal with Sq < Sk is aligned to the bottom right: the 128 rows see
    # (almost) every key
    c = Case(1, 1, 128, LONG, 64, 64, kind, lists=lists, sparse=(128, 512) if lists else None)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    assert_no_device_error()
    p = c.problem(0, 0)
    o_ref, l_ref = p.forward()
    check_out(f64(o[0, 0]), o_ref)
    check_lse(f64(lse[0, 0]), l_ref)
    dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, 0])
    check_grad(f64(dq[0, 0]), dq_r, "dQ")
    check_grad(f64(dk[0, 0]), dk_r, "dK")
    check_grad(f64(dv[0, 0]), dv_r, "dV")


def test_key_tile_under_more_than_1024_query_tiles():
    c = Case(1, 1, LONG, 128, 64, 64, "none", lists=False, sparse=None)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    assert_no_device_error()
    p = c.problem(0, 0)
    o_ref, l_ref = p.forward()
    check_out(f64(o[0, 0]), o_ref)
    check_lse(f64(lse[0, 0]), l_ref)
    dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, 0])
    check_grad(f64(dq[0, 0]), dq_r, "dQ")
    check_grad(f64(dk[0, 0]), dk_r, "dK")
    check_grad(f64(dv[0, 0]), dv_r, "dV")


def test_gathered_row_over_more_than_1024_compact_key_tiles():
    # dynamic top-k keeping all but 256 of the keys: the compact (kept) key
    # tiles of the one query tile number 1036
    c = Case(1, 1, 128, LONG + 256, 64, 64, "dynamic", topk=LONG, gather=True, sparse=(128, 128))
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    assert_no_device_error()
    p = c.problem(0, 0)
    o_ref, l_ref = p.forward()
    check_out(f64(o[0, 0]), o_ref)
    check_lse(f64(lse[0, 0]), l_ref)
    dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, 0])
    check_grad(f64(dq[0, 0]), dq_r, "dQ")
    check_grad(f64(dk[0, 0]), dk_r, "dK")
    check_grad(f64(dv[0, 0]), dv_r, "dV")


def test_pair_dkdv_under_more_than_1024_query_tiles():
    # the CTA-pair dK/dV kernel: one pair of key tiles, 1036 query tiles
    c = Case(1, 1, LONG, 256, 128, 128, "none", lists=False, sparse=None)
    o, lse = c.fwd()
    prev = ga.set_dkdv_cta_pair(1)
    try:
        dq, dk, dv = c.bwd(o, lse)
    finally:
        ga.set_dkdv_cta_pair(prev)
    assert_no_device_error()
    dq_r, dk_r, dv_r, _ = c.problem(0, 0).backward(c.h["do"][0, 0])
    check_grad(f64(dq[0, 0]), dq_r, "dQ")
    check_grad(f64(dk[0, 0]), dk_r, "dK")
    check_grad(f64(dv[0, 0]), dv_r, "dV")
