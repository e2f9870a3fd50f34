"""Parity at the workloads' full sizes, in the launch configuration bench.py
times: the GPU computes every output; the oracle recomputes sampled rows /
key columns / heads one by one (each row or column is defined on its own),
and the block lists are compared bit-exactly in full."""
import numpy as np
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga
from block_sparse_attention_tma_gb300.synth import make_device_inputs
from helpers import Case, check_dbias, check_grad, check_lse, check_out, f64, assert_no_device_error
from oracle import attention as orc

pytestmark = pytest.mark.gpu

LIST_NAMES = ["q_mask_cnt", "q_mask_idx", "q_full_cnt", "q_full_idx",
              "k_mask_cnt", "k_mask_idx", "k_full_cnt", "k_full_idx"]


def sample_idx(n, k=96, seed=0):
    rng = np.random.default_rng(seed)
    picks = set([0, 1, 127, 128, n // 2, n - 129, n - 2, n - 1])
    picks |= set(rng.choice(n, size=min(k, n), replace=False).tolist())
    return np.array(sorted(p for p in picks if 0 <= p < n))


def lists_equal_headwise(c, ref_by_head, B, H):
    for n in LIST_NAMES:
        g = c.lists.tensors[n].cpu().numpy()
        for b in range(B):
            for h in range(H):
                ref = ref_by_head(b, h)[n][0, 0]
                got = g.reshape((B, H) + ref.shape)[b, h]
                assert np.array_equal(got, ref), (n, b, h)


def check_rows_cols(c, b, h, rows, cols, o, lse, grads=None):
    p = c.problem(b, h)
    o_ref, l_ref = p.forward(rows)
    check_out(f64(o[b, h])[rows], o_ref)
    check_lse(f64(lse[b, h])[rows], l_ref)
    if grads is not None:
        dq, dk, dv = grads
        dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][b, h], rows=rows, cols=cols)
        # relative-to-max over the sampled entries
        check_grad(f64(dq[b, h])[rows], dq_r, "dQ")
        check_grad(f64(dk[b, h])[cols], dk_r, "dK")
        check_grad(f64(dv[b, h])[cols], dv_r, "dV")


def test_tiny_fp32_causal_full():
    c = Case(1, 1, 128, 128, 64, 64, "causal", dtype="fp32", sparse=(128, 128))
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    p = c.problem(0, 0)
    o_ref, l_ref = p.forward()
    check_out(f64(o[0, 0]), o_ref, fp32=True)
    check_lse(f64(lse[0, 0]), l_ref, fp32=True)
    dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, 0])
    for g, r, n in ((dq, dq_r, "dQ"), (dk, dk_r, "dK"), (dv, dv_r, "dV")):
        check_grad(f64(g[0, 0]), r, n, fp32=True)


@pytest.mark.parametrize("kind,extra", [("causal", {}), ("sliding", dict(window=512))])
def test_dense_masked_2x8x2048_d64(kind, extra):
    B, H, S = 2, 8, 2048
    c = Case(B, H, S, S, 64, 64, kind, sparse=(128, 128), **extra)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    for b in range(B):
        for h in range(H):
            p = c.problem(b, h)
            o_ref, l_ref = p.forward()
            check_out(f64(o[b, h]), o_ref)
            check_lse(f64(lse[b, h]), l_ref)
    for (b, h) in ((0, 0), (1, 7)):
        dq_r, dk_r, dv_r, _ = c.problem(b, h).backward(c.h["do"][b, h])
        check_grad(f64(dq[b, h]), dq_r, "dQ")
        check_grad(f64(dk[b, h]), dk_r, "dK")
        check_grad(f64(dv[b, h]), dv_r, "dV")


@pytest.mark.parametrize("D", [32, 64])
def test_dynamic_topk_1x16x8192(D):
    B, H, S = 1, 16, 8192
    c = Case(B, H, S, S, D, D, "dynamic", topk=2048, sparse=(128, 128))
    torch.cuda.synchronize()
    lists_equal_headwise(c, lambda b, h: orc.block_lists(
        1, 1, S, S, dict(kind=orc.DYNAMIC_TOPK, topk=2048, key_bias=c.od["key_bias"][b:b + 1, h:h + 1]), 128, 128),
        B, H)
    bits = orc.keep_bits(c.od["key_bias"], 2048)
    got = c.lists.tensors["keep_bits"].cpu().numpy().view(np.uint32).reshape(bits.shape)
    assert np.array_equal(got, bits)
    idx = orc.keep_index(c.od["key_bias"], 2048)
    got = c.lists.tensors["keep_idx"].cpu().numpy().reshape(idx.shape)
    assert np.array_equal(got, idx)
    # the gathered path (kept keys only), as bench.py runs it
    o, lse = c.fwd()
    db = c.dbias_buffer()
    dq, dk, dv = c.bwd(o, lse, dkey_bias=db)
    torch.cuda.synchronize()
    assert_no_device_error()
    rows, cols = sample_idx(S, seed=1), sample_idx(S, seed=2)
    for h in (0, 9):
        check_rows_cols(c, 0, h, rows, cols, o, lse, (dq, dk, dv) if h == 0 else None)
    check_dbias(f64(db[0, 0])[cols], c.problem(0, 0).dkey_bias(c.h["do"][0, 0], cols))
    assert np.all(np.isfinite(f64(db)))


@pytest.mark.parametrize("kind,extra", [("causal", {}), ("sliding", {}), ("block_diag", dict(block_size=1024)),
                                        ("prefix_lm", dict(prefix_len=2048))])
def test_block_sparse_mla_1x16x16384(kind, extra):
    B, H, S = 1, 16, 16384
    c = Case(B, H, S, S, 192, 128, kind, sparse=(256, 512), slope=0.01, **extra)
    torch.cuda.synchronize()
    # closed-form masks do not depend on (b, h): one reference head serves all
    ref = orc.block_lists(1, 1, S, S, c.od, 256, 512)
    lists_equal_headwise(c, lambda b, h: ref, B, H)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    rows, cols = sample_idx(S, seed=3), sample_idx(S, seed=4)
    # heads 0 and 5 with gradients (the heaviest-first tile order launches the
    # first and last heads in different waves), head 15 forward only
    check_rows_cols(c, 0, 0, rows, cols, o, lse, (dq, dk, dv))
    check_rows_cols(c, 0, 5, rows, cols, o, lse, (dq, dk, dv))
    check_rows_cols(c, 0, 15, rows, cols, o, lse)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16])
def test_splitkv_decode_32x32x65536(n):
    B, H, Sk, D = 32, 32, 65536, 128
    x = make_device_inputs(B, H, 1, Sk, D, D, "bf16", seed=42, dout=False)
    o, lse = ga.attn_fwd_splitkv(x["q"], x["k"], x["v"], 0.0, None, n)
    torch.cuda.synchronize()
    assert_no_device_error()
    for (b, h) in ((0, 0), (3, 17), (31, 31), (17, 5)):
        p = orc.Problem(f64(x["q"][b, h]), f64(x["k"][b, h]), f64(x["v"][b, h]))
        o_ref, l_ref = p.forward()
        check_out(f64(o[b, h]), o_ref)
        check_lse(f64(lse[b, h]), l_ref)
    del x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("Hkv,paged,n", [(8, True, 4), (1, False, 4), (4, False, 1)])
def test_gqa_decode_32x32x65536(Hkv, paged, n):
    # grouped-query decode at the decode workload's size: packed tensor-core
    # path, dense or over a shuffled 256-key page pool with per-sequence lengths
    B, H, Sk, D, page = 32, 32, 65536, 128, 256
    x = make_device_inputs(B, H, 1, Sk, D, D, "bf16", seed=42, dout=False, Hkv=Hkv)
    G = H // Hkv
    if paged:
        npg = Sk // page
        kc = x["k"].view(B, Hkv, npg, page, D).permute(0, 2, 1, 3, 4).reshape(B * npg, Hkv, page, D)
        vc = x["v"].view(B, Hkv, npg, page, D).permute(0, 2, 1, 3, 4).reshape(B * npg, Hkv, page, D)
        perm = torch.randperm(B * npg, generator=torch.Generator().manual_seed(3)).cuda()
        kpool = torch.empty_like(kc)
        vpool = torch.empty_like(vc)
        kpool[perm] = kc
        vpool[perm] = vc
        del kc, vc
        table = perm.view(B, npg).to(torch.int32).contiguous()
        rng = np.random.default_rng(5)
        lens = rng.integers(1, Sk + 1, size=B)
        lens[0], lens[1] = Sk, 1
        seqlens = torch.from_numpy(lens.astype(np.int32)).cuda()
        o, lse = ga.attn_fwd_splitkv_paged(x["q"], kpool, vpool, table, seqlens, 0.0, None, n)
    else:
        lens = np.full(B, Sk)
        o, lse = ga.attn_fwd_splitkv(x["q"], x["k"], x["v"], 0.0, None, n)
    torch.cuda.synchronize()
    assert_no_device_error()
    for (b, h) in ((0, 0), (1, 5), (7, 31), (20, 17), (31, 8)):
        L = int(lens[b])
        hk = h // G
        p = orc.Problem(f64(x["q"][b, h]), f64(x["k"][b, hk, :L]), f64(x["v"][b, hk, :L]))
        o_ref, l_ref = p.forward()
        check_out(f64(o[b, h]), o_ref)
        check_lse(f64(lse[b, h]), l_ref)
    del x
    torch.cuda.empty_cache()


def test_gqa_16k_head_grouped_order():
    """Grouped-query attention at a size where the prefill kernels take the
    heads in groups (the dK/dV grid's per-key/value-head Q + dO bytes exceed
    half the L2): 1 x 8 query heads on 2 key/value heads x 16384, 128/128,
    causal, 256 x 512 lists. Sampled rows of O / LSE / dQ for query heads of
    both groups, and sampled key columns of dK / dV for both key/value heads,
    each the sum over its four query heads."""
    B, H, Hkv, S, D = 1, 8, 2, 16384, 128
    c = Case(B, H, S, S, D, D, "causal", sparse=(256, 512), Hkv=Hkv)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    G = H // Hkv
    rows, cols = sample_idx(S, k=48, seed=5), sample_idx(S, k=48, seed=6)
    for h in (0, 5):
        p = c.problem(0, h)
        o_ref, l_ref = p.forward(rows)
        check_out(f64(o[0, h])[rows], o_ref)
        check_lse(f64(lse[0, h])[rows], l_ref)
        dq_r, _, _, _ = p.backward(c.h["do"][0, h], rows=rows, cols=cols[:1])
        check_grad(f64(dq[0, h])[rows], dq_r, "dQ")
    for hk in range(Hkv):
        dk_sum = dv_sum = 0
        for g in range(G):
            h = hk * G + g
            _, dk_r, dv_r, _ = c.problem(0, h).backward(c.h["do"][0, h], rows=rows[:1], cols=cols)
            dk_sum, dv_sum = dk_sum + dk_r, dv_sum + dv_r
        check_grad(f64(dk[0, hk])[cols], dk_sum, "dK")
        check_grad(f64(dv[0, hk])[cols], dv_sum, "dV")
