"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test pins one part of the definition with something independent of it:
closed forms, special cases, a library routine (torch CPU float64 SDPA +
autograd), central finite differences, brute-force rank counts, and the
algebra of the split-KV merge. No GPU is needed.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from conftest import read_golden

KINDS = {
    "none": dict(kind=A.NONE),
    "causal": dict(kind=A.CAUSAL),
    "sliding": dict(kind=A.SLIDING, window_left=5),
    "block_diag": dict(kind=A.BLOCK_DIAG, block_size=8),
    "prefix_lm": dict(kind=A.PREFIX_LM, prefix_len=6),
    "dynamic": dict(kind=A.DYNAMIC_TOPK, topk=9),
    "mini_causal": dict(kind=A.MINI_CAUSAL, block_size=4),
    # an arbitrary predicate: the allowed pairs of a fixed random table
    "table": dict(kind=A.TABLE, table=np.random.default_rng(99).random((64, 64)) < 0.6),
}


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _problem(rng, sq, sk, dqk, dv, spec, bias=False, slope=0.0, softcap=0.0):
    q, k, v = _rand(rng, sq, dqk), _rand(rng, sk, dqk), _rand(rng, sk, dv)
    kb = _rand(rng, sk) if (bias or spec["kind"] == A.DYNAMIC_TOPK) else None
    if spec["kind"] == A.TABLE:  # the table's top-left Sq x Sk corner
        spec = dict(spec, table=spec["table"][:sq, :sk])
    return A.Problem(q, k, v, key_bias=kb, rel_bias_slope=slope, softcap=softcap, **spec)


@pytest.mark.parametrize("name", list(KINDS))
@pytest.mark.parametrize("shape", [(19, 19), (13, 29), (29, 13)])
def test_rows_sum_to_one(name, shape):
    rng = np.random.default_rng(1)
    p = _problem(rng, *shape, 8, 6, KINDS[name], bias=True, slope=0.03, softcap=3.0)
    P, lse = p.probs(np.arange(p.sq))
    live = np.isfinite(lse)
    assert np.all(np.abs(P[live].sum(1) - 1.0) < 1e-12)
    assert np.all(P[~live] == 0.0)
    # P is zero exactly where the mask says so
    m = p.mask(np.arange(p.sq), np.arange(p.sk))
    assert np.all(P[~m] == 0.0)


@pytest.mark.parametrize("name", list(KINDS))
def test_constant_v_gives_constant_output(name):
    rng = np.random.default_rng(2)
    p = _problem(rng, 23, 31, 8, 5, KINDS[name], bias=True, slope=0.02)
    p.v[:] = 0.375
    o, lse = p.forward()
    live = np.isfinite(lse)
    assert np.all(np.abs(o[live] - 0.375) < 1e-13)
    assert np.all(o[~live] == 0.0)


@pytest.mark.parametrize("name", ["none", "causal", "sliding", "block_diag", "prefix_lm"])
def test_zero_q_gives_mean_of_allowed_values(name):
    rng = np.random.default_rng(3)
    p = _problem(rng, 17, 26, 8, 4, KINDS[name])
    p.q[:] = 0.0
    o, lse = p.forward()
    m = p.mask(np.arange(p.sq), np.arange(p.sk))
    for i in range(p.sq):
        n = m[i].sum()
        if n == 0:
            assert lse[i] == -np.inf and np.all(o[i] == 0)
            continue
        assert np.allclose(o[i], p.v[m[i]].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[i] - math.log(n)) < 1e-13


def test_causal_row_zero_and_single_key():
    rng = np.random.default_rng(4)
    p = _problem(rng, 9, 9, 8, 4, KINDS["causal"])
    o, lse = p.forward()
    assert np.allclose(o[0], p.v[0], atol=1e-15)
    assert abs(lse[0] - p.scale * float(p.q[0] @ p.k[0])) < 1e-13
    p1 = _problem(rng, 6, 1, 8, 4, KINDS["none"])
    o1, lse1 = p1.forward()
    assert np.allclose(o1, np.broadcast_to(p1.v[0], o1.shape), atol=1e-15)
    assert np.allclose(lse1, p1.scale * (p1.q @ p1.k[0]), atol=1e-13)


def test_lse_shift_invariance():
    rng = np.random.default_rng(5)
    p = _problem(rng, 15, 21, 8, 4, KINDS["prefix_lm"], bias=True, slope=0.01)
    o, lse = p.forward()
    p.key_bias = p.key_bias + 2.5
    o2, lse2 = p.forward()
    assert np.allclose(o, o2, atol=1e-13)
    assert np.allclose(lse2 - lse, 2.5, atol=1e-12)


def test_fully_masked_rows_convention():
    # block-diagonal with Sq > Sk: rows with i + (Sk - Sq) < 0 see no key
    rng = np.random.default_rng(6)
    p = _problem(rng, 12, 5, 4, 3, dict(kind=A.BLOCK_DIAG, block_size=4))
    o, lse = p.forward()
    dead = (np.arange(12) + (5 - 12)) < 0
    assert dead.sum() == 7
    assert np.all(lse[dead] == -np.inf) and np.all(o[dead] == 0.0)
    dq, dk, dv, _ = p.backward(_rand(rng, 12, 3))
    assert np.all(dq[dead] == 0.0)
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def _loss(p, do):
    o, _ = p.forward()
    return float(np.sum(o * do))


@pytest.mark.parametrize("name", list(KINDS))
@pytest.mark.parametrize("extras", [dict(), dict(bias=True, slope=0.05, softcap=2.0)])
@pytest.mark.parametrize("shape", [(5, 7), (7, 5)])
def test_gradients_match_finite_differences(name, extras, shape):
    rng = np.random.default_rng(7)
    p = _problem(rng, *shape, 4, 3, KINDS[name], **extras)
    do = _rand(rng, p.sq, p.dv)
    dq, dk, dv, _ = p.backward(do)
    h = 1e-6
    for arr, grad in ((p.q, dq), (p.k, dk), (p.v, dv)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            x0 = arr[idx]
            arr[idx] = x0 + h
            lp = _loss(p, do)
            arr[idx] = x0 - h
            lm = _loss(p, do)
            arr[idx] = x0
            num[idx] = (lp - lm) / (2 * h)
        scale = max(1.0, np.abs(num).max())
        assert np.abs(num - grad).max() / scale < 1e-6


@pytest.mark.parametrize("name", list(KINDS))
@pytest.mark.parametrize("extras", [dict(), dict(slope=0.05, softcap=2.0)])
def test_key_bias_gradient_matches_finite_differences(name, extras):
    # L = <dO, O> as a function of each key bias (the dynamic keep set is fixed
    # at construction, so the perturbation moves the scores only)
    rng = np.random.default_rng(17)
    p = _problem(rng, 6, 9, 4, 3, KINDS[name], bias=True, **extras)
    do = _rand(rng, p.sq, p.dv)
    g = p.dkey_bias(do)
    h = 1e-6
    num = np.zeros(p.sk)
    for j in range(p.sk):
        x0 = p.key_bias[j]
        p.key_bias[j] = x0 + h
        lp = _loss(p, do)
        p.key_bias[j] = x0 - h
        lm = _loss(p, do)
        p.key_bias[j] = x0
        num[j] = (lp - lm) / (2 * h)
    assert np.abs(num - g).max() / max(1.0, np.abs(num).max()) < 1e-6
    # a subset of columns is the same numbers
    cols = np.array([0, 4, 8])
    assert np.array_equal(p.dkey_bias(do, cols), g[cols])


@pytest.mark.parametrize("name", list(KINDS))
def test_key_bias_gradient_sums_to_zero_and_matches_autograd(name):
    # sum_j dL/dkb_j = sum_i sum_j P_ij (dP_ij - D_i) = 0 for every live row,
    # softcap or not (the cap acts before the bias); keys no query sees get 0
    rng = np.random.default_rng(18)
    p = _problem(rng, 23, 31, 8, 5, KINDS[name], bias=True, slope=0.03, softcap=1.5)
    do = _rand(rng, p.sq, p.dv)
    g = p.dkey_bias(do)
    assert abs(g.sum()) < 1e-12
    unused = ~p.mask(np.arange(p.sq), np.arange(p.sk)).any(0)
    assert np.all(g[unused] == 0.0)
    # torch float64 autograd through an explicit softmax with the bias as a leaf
    rows, cols = np.arange(p.sq), np.arange(p.sk)
    m = torch.tensor(p.mask(rows, cols))
    kb = torch.tensor(p.key_bias, requires_grad=True)
    r = p.scale * torch.tensor(p.q) @ torch.tensor(p.k).T
    r = p.softcap * torch.tanh(r / p.softcap)
    s = r + p.rel_bias_slope * torch.tensor(rows[:, None] - cols[None, :], dtype=torch.float64) + kb[None, :]
    s = torch.where(m, s, torch.tensor(-math.inf, dtype=torch.float64))
    live = m.any(1)
    pr = torch.where(live[:, None], torch.softmax(torch.where(live[:, None], s, torch.zeros_like(s)), 1)
                     * m, torch.zeros_like(s))
    out = pr @ torch.tensor(p.v)
    out.backward(torch.tensor(do))
    assert np.allclose(g, kb.grad.numpy(), atol=1e-11)


def test_keep_index_lists_kept_keys_ascending():
    rng = np.random.default_rng(19)
    kb = np.round(rng.standard_normal((2, 2, 45)) * 2) / 2  # ties
    for k in (0, 1, 10, 45, 60):
        idx = A.keep_index(kb, k)
        assert idx.shape == (2, 2, 45) and idx.dtype == np.int32
        for b in range(2):
            for h in range(2):
                row = kb[b, h]
                # brute-force rank count, independent of the lexsort in topk_keep
                kept = [j for j in range(45)
                        if sum(1 for i in range(45) if row[i] > row[j] or (row[i] == row[j] and i < j)) < k]
                n = len(kept)
                assert n == min(k, 45)
                assert idx[b, h, :n].tolist() == kept  # ascending by construction of the list above
                assert np.all(idx[b, h, n:] == 0)


@pytest.mark.parametrize("name", list(KINDS))
def test_backward_invariants(name):
    rng = np.random.default_rng(8)
    p = _problem(rng, 21, 33, 8, 6, KINDS[name], bias=True)
    do = _rand(rng, p.sq, p.dv)
    rows = np.arange(p.sq)
    P, lse = p.probs(rows)
    o, _ = p.forward()
    dP = do @ p.v.T
    D = np.sum(do * o, axis=1)
    assert np.allclose(D, np.sum(P * dP, axis=1), atol=1e-12)
    dS = P * (dP - D[:, None])
    assert np.all(np.abs(dS.sum(1)) < 1e-12)
    dq, dk, dv, d_all = p.backward(do)
    assert np.allclose(d_all, D, atol=1e-13)
    # dV rows of keys no query attends to are zero
    m = p.mask(rows, np.arange(p.sk))
    unused = ~m.any(0)
    assert np.all(dv[unused] == 0) and np.all(dk[unused] == 0)


@pytest.mark.parametrize("name", list(KINDS))
def test_matches_torch_float64_sdpa_and_autograd(name):
    rng = np.random.default_rng(9)
    sq, sk, dqk, dv = 37, 53, 16, 8
    p = _problem(rng, sq, sk, dqk, dv, KINDS[name], bias=True, slope=0.02)
    do = _rand(rng, sq, dv)
    rows, cols = np.arange(sq), np.arange(sk)
    m = p.mask(rows, cols)
    assert m.any(1).all()  # torch's SDPA has no convention for empty rows
    add = p.rel_bias_slope * (rows[:, None] - cols[None, :]) + p.key_bias[None, :]
    add = np.where(m, add, -np.inf)
    tq = torch.tensor(p.q, requires_grad=True)
    tk = torch.tensor(p.k, requires_grad=True)
    tv = torch.tensor(p.v, requires_grad=True)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], attn_mask=torch.tensor(add)[None], scale=p.scale)[0]
    out.backward(torch.tensor(do))
    o, lse = p.forward()
    dq, dk, dvv, _ = p.backward(do)
    assert np.allclose(o, out.detach().numpy(), atol=1e-12)
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dvv, tv.grad.numpy(), atol=1e-11)
    ref_lse = torch.logsumexp(torch.tensor(p.scale * (p.q @ p.k.T) + add), dim=1).numpy()
    assert np.allclose(lse, ref_lse, atol=1e-12)


def test_grouped_query_reading_matches_torch_enable_gqa():
    # GQA reading: query head h reads key/value head h // (H / Hkv), and the
    # gradient of a key/value head sums over its query heads. Pinned against
    # torch's float64 SDPA with enable_gqa=True and autograd (a library routine).
    rng = np.random.default_rng(21)
    H, Hkv, sq, sk, d = 6, 2, 19, 23, 8
    G = H // Hkv
    q, k, v = _rand(rng, H, sq, d), _rand(rng, Hkv, sk, d), _rand(rng, Hkv, sk, d)
    do = _rand(rng, H, sq, d)
    rows, cols = np.arange(sq), np.arange(sk)
    m = A.allowed(A.CAUSAL, sq, sk, rows, cols)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], attn_mask=torch.tensor(m)[None, None], enable_gqa=True)[0]
    out.backward(torch.tensor(do))
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(H):
        p = A.Problem(q[h], k[h // G], v[h // G], kind=A.CAUSAL)
        o, _ = p.forward()
        assert np.allclose(o, out[h].detach().numpy(), atol=1e-12)
        dq_h, dk_h, dv_h, _ = p.backward(do[h])
        assert np.allclose(dq_h, tq.grad[h].numpy(), atol=1e-11)
        dk[h // G] += dk_h
        dv[h // G] += dv_h
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_mini_causal_reading():
    # causal inside blocks: a per-element brute force of the reading, its
    # closed-form pair count, and the two limits (one block = causal; blocks
    # of one key = the diagonal only)
    for sq, sk, bs in ((16, 16, 4), (13, 21, 5), (21, 13, 3)):
        m = A.allowed(A.MINI_CAUSAL, sq, sk, np.arange(sq), np.arange(sk), block_size=bs)
        for i in range(sq):
            a = i + sk - sq
            for j in range(sk):
                assert m[i, j] == (j <= a and a // bs == j // bs)
    S, bs = 1024, 128
    assert A.pair_count(S, S, dict(kind=A.MINI_CAUSAL, block_size=bs)) == (S // bs) * bs * (bs + 1) // 2
    rows, cols = np.arange(40), np.arange(40)
    assert np.array_equal(A.allowed(A.MINI_CAUSAL, 40, 40, rows, cols, block_size=64),
                          A.allowed(A.CAUSAL, 40, 40, rows, cols))
    assert np.array_equal(A.allowed(A.MINI_CAUSAL, 40, 40, rows, cols, block_size=1), np.eye(40, dtype=bool))


def test_table_mask_reproduces_the_closed_form_kinds():
    # a table holding another kind's element mask gives that kind's result
    # exactly (same mask matrix, same arithmetic), lists included
    rng = np.random.default_rng(23)
    sq, sk = 37, 45
    q, k, v, do = _rand(rng, sq, 8), _rand(rng, sk, 8), _rand(rng, sk, 4), _rand(rng, sq, 4)
    rows, cols = np.arange(sq), np.arange(sk)
    for spec in (dict(kind=A.CAUSAL), dict(kind=A.SLIDING, window_left=6), dict(kind=A.MINI_CAUSAL, block_size=8)):
        tab = A.allowed(spec["kind"], sq, sk, rows, cols, window_left=spec.get("window_left", -1),
                        block_size=spec.get("block_size", 0))
        p1 = A.Problem(q, k, v, **spec)
        p2 = A.Problem(q, k, v, kind=A.TABLE, table=tab)
        o1, l1 = p1.forward()
        o2, l2 = p2.forward()
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
        g1, g2 = p1.backward(do), p2.backward(do)
        for a, b in zip(g1, g2):
            assert np.array_equal(a, b)
        L1 = A.block_lists(1, 1, sq, sk, spec, 128, 128)
        L2 = A.block_lists(1, 1, sq, sk, dict(kind=A.TABLE, table=tab), 128, 128)
        for n in L1:
            assert np.array_equal(L1[n], L2[n])
    # per-head tables pick the head's own matrix
    t = rng.random((1, 2, sq, sk)) < 0.5
    L = A.block_lists(1, 2, sq, sk, dict(kind=A.TABLE, table=t), 128, 128)
    assert L["q_mask_cnt"].shape == (1, 2, 1)


def test_topk_matches_brute_force_ranks_with_ties():
    rng = np.random.default_rng(10)
    for sk, k in ((40, 7), (64, 64), (33, 50), (50, 0), (1, 1)):
        b = np.round(rng.standard_normal(sk) * 2) / 2  # many ties
        keep = A.topk_keep(b, k)
        for j in range(sk):
            rank = sum(1 for i in range(sk) if b[i] > b[j] or (b[i] == b[j] and i < j))
            assert keep[j] == (rank < k)
    # plain python sort as a second opinion
    b = rng.standard_normal(100).astype(np.float32).astype(np.float64)
    order = sorted(range(100), key=lambda j: (-b[j], j))[:10]
    assert set(np.nonzero(A.topk_keep(b, 10))[0]) == set(order)


def test_keep_bits_packing():
    rng = np.random.default_rng(11)
    kb = rng.standard_normal((1, 2, 70))
    bits = A.keep_bits(kb, 20)
    for h in range(2):
        keep = A.topk_keep(kb[0, h], 20)
        unpacked = [(int(bits[0, h, j // 32]) >> (j % 32)) & 1 for j in range(70)]
        assert unpacked == [int(x) for x in keep]
        assert int(bits[0, h, 2]) >> 6 == 0  # bits past Sk are zero


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("name", ["none", "causal"])
def test_split_merge_equals_unsplit(n, name):
    rng = np.random.default_rng(12)
    p = _problem(rng, 3, 700, 8, 5, KINDS[name])
    o_parts, lse_parts = p.split_partials(n)
    o, lse = A.combine_splits(o_parts, lse_parts)
    o_ref, lse_ref = p.forward()
    assert np.allclose(o, o_ref, atol=1e-12) and np.allclose(lse, lse_ref, atol=1e-12)
    bounds = A.Problem.split_bounds(700, n)
    assert bounds[0][0] == 0 and bounds[-1][1] == 700
    assert all(b0 % 128 == 0 for b0, b1 in bounds if b1 > b0)


def test_split_merge_arbitrary_partition_and_empty_splits():
    rng = np.random.default_rng(13)
    p = _problem(rng, 4, 50, 8, 5, KINDS["none"])
    # 16 splits of 50 keys at 128-key granularity: all but the first are empty
    o_parts, lse_parts = p.split_partials(16)
    assert np.all(np.isinf(lse_parts[1:]))
    o, lse = A.combine_splits(o_parts, lse_parts)
    o_ref, lse_ref = p.forward()
    assert np.allclose(o, o_ref, atol=1e-12) and np.allclose(lse, lse_ref, atol=1e-12)
    # hand-made partition through the merge rule
    parts = [(0, 11), (11, 12), (12, 50)]
    ol, ll = [], []
    for a, b in parts:
        sub = A.Problem(p.q, p.k[a:b], p.v[a:b], scale=p.scale)
        oo, l_ = sub.forward()
        ol.append(oo)
        ll.append(l_)
    o2, lse2 = A.combine_splits(np.stack(ol), np.stack(ll))
    assert np.allclose(o2, o_ref, atol=1e-12) and np.allclose(lse2, lse_ref, atol=1e-12)


def _tri(n):
    return n * (n + 1) // 2


def test_pair_counts_closed_forms():
    S = 2048
    assert A.pair_count(S, S, dict(kind=A.CAUSAL)) == _tri(S)
    W = 512
    # keys j in [i - W, i]: i + 1 keys for i < W, W + 1 after
    assert A.pair_count(S, S, dict(kind=A.SLIDING, window_left=W)) == _tri(W) + (S - W) * (W + 1)
    assert A.pair_count(S, S, dict(kind=A.BLOCK_DIAG, block_size=256)) == (S // 256) * 256 * 256
    P = 300
    # row i sees max(P, i + 1) keys
    assert A.pair_count(S, S, dict(kind=A.PREFIX_LM, prefix_len=P)) == P * P + (_tri(S) - _tri(P))
    # Sq != Sk, causal bottom-right: row i sees min(Sk, i + Sk - Sq + 1) keys (>= 0)
    sq, sk = 300, 1000
    assert A.pair_count(sq, sk, dict(kind=A.CAUSAL)) == sum(min(sk, i + sk - sq + 1) for i in range(sq))
    # 2 x 8 heads at 2048, causal: the dense masked workload's pair count
    assert 16 * A.pair_count(2048, 2048, dict(kind=A.CAUSAL)) == 33_570_816


def test_window_rule_fixture():
    for sq, sk, w in read_golden("fa_pr2661_window_rule.txt"):
        assert max(64, min(int(sq), int(sk)) // 3) == int(w)


def test_block_lists_closed_form_causal_256x512():
    S = 4096
    lists = A.block_lists(1, 1, S, S, dict(kind=A.CAUSAL), 256, 512)
    nqb, nkb = S // 256, S // 512
    for r in range(nqb):
        full = [c for c in range(nkb) if 512 * c + 511 <= 256 * r]
        part = [c for c in range(nkb) if 512 * c <= 256 * r + 255 and c not in full]
        assert lists["q_full_cnt"][0, 0, r] == len(full)
        assert list(lists["q_full_idx"][0, 0, r, :len(full)]) == full
        assert lists["q_mask_cnt"][0, 0, r] == len(part)
        assert list(lists["q_mask_idx"][0, 0, r, :len(part)]) == part
        assert np.all(lists["q_mask_idx"][0, 0, r, len(part):] == 0)


def test_block_lists_block_diag_and_ragged_edge():
    # 1000 x 1000 at 256 x 512 blocks, block-diagonal 256: the last row block
    # and last column block are cut by the sequence end and never full.
    lists = A.block_lists(1, 1, 1000, 1000, dict(kind=A.BLOCK_DIAG, block_size=256), 256, 512)
    # q-block r covers diagonal block r; k-block c covers diag blocks 2c, 2c+1
    for r in range(4):
        c = r // 2
        assert lists["q_mask_cnt"][0, 0, r] == 1 and lists["q_mask_idx"][0, 0, r, 0] == c
        assert lists["q_full_cnt"][0, 0, r] == 0  # half of each 512-wide block is off-diagonal
    # at 256 x 256 blocks the diagonal blocks are full, except the cut last one
    lists = A.block_lists(1, 1, 1000, 1000, dict(kind=A.BLOCK_DIAG, block_size=256), 256, 256)
    assert list(lists["q_full_cnt"][0, 0]) == [1, 1, 1, 0]
    assert list(lists["q_mask_cnt"][0, 0]) == [0, 0, 0, 1]
    lists = A.block_lists(1, 1, 1000, 1000, dict(kind=A.NONE), 256, 256)
    assert list(lists["q_full_cnt"][0, 0]) == [3, 3, 3, 0]
    assert list(lists["q_mask_cnt"][0, 0]) == [1, 1, 1, 4]


@pytest.mark.parametrize("row", read_golden("fa_pr2661_fuzz_cases.txt"))
def test_fwd_and_bwd_lists_describe_the_same_blocks(row):
    seed, sq, sk, dqk, dv, stm, stn, name = row
    sq, sk, stm, stn = int(sq), int(sk), int(stm), int(stn)
    spec = {"causal": dict(kind=A.CAUSAL),
            "sliding_window": dict(kind=A.SLIDING, window_left=max(64, min(sq, sk) // 3)),
            "block_diagonal": dict(kind=A.BLOCK_DIAG, block_size=256),
            "mini_causal": dict(kind=A.MINI_CAUSAL, block_size=256)}[name]
    L = A.block_lists(1, 1, sq, sk, spec, stm, stn)
    fwd = {(r, int(L["q_mask_idx"][0, 0, r, t]), "m") for r in range(L["q_mask_cnt"].shape[2])
           for t in range(L["q_mask_cnt"][0, 0, r])}
    fwd |= {(r, int(L["q_full_idx"][0, 0, r, t]), "f") for r in range(L["q_full_cnt"].shape[2])
            for t in range(L["q_full_cnt"][0, 0, r])}
    bwd = {(int(L["k_mask_idx"][0, 0, c, t]), c, "m") for c in range(L["k_mask_cnt"].shape[2])
           for t in range(L["k_mask_cnt"][0, 0, c])}
    bwd |= {(int(L["k_full_idx"][0, 0, c, t]), c, "f") for c in range(L["k_full_cnt"].shape[2])
            for t in range(L["k_full_cnt"][0, 0, c])}
    assert fwd == bwd
    # every allowed pair lies in a listed block; every full block has all pairs
    m = A.allowed(spec["kind"], sq, sk, np.arange(sq), np.arange(sk),
                  window_left=spec.get("window_left", -1), block_size=spec.get("block_size", 0))
    for i, j in zip(*np.nonzero(m)):
        assert (i // stm, j // stn, "m") in fwd or (i // stm, j // stn, "f") in fwd
    for (r, c, kind) in fwd:
        blk = m[r * stm:(r + 1) * stm, c * stn:(c + 1) * stn]
        assert blk.any()
        if kind == "f":
            assert blk.all() and blk.shape == (stm, stn)
