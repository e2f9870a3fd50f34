"""GPU parity: every step of the hot path through the C ABI against the fp64
oracle on the same seeded inputs (element by element at sizes the oracle
finishes in seconds, spanning several 128-tiles and a ragged tail)."""
import numpy as np
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga
from conftest import golden_setup, read_golden
from helpers import Case, check_dbias, check_grad, check_lse, check_out, f64, assert_no_device_error, make_table
from oracle import attention as orc

pytestmark = pytest.mark.gpu

LIST_NAMES = ["q_mask_cnt", "q_mask_idx", "q_full_cnt", "q_full_idx",
              "k_mask_cnt", "k_mask_idx", "k_full_cnt", "k_full_idx"]


def lists_equal(c, B, H, Sq, Sk, sm, sn):
    ref = orc.block_lists(B, H, Sq, Sk, c.od, sm, sn)
    for n in LIST_NAMES:
        g = c.lists.tensors[n].cpu().numpy().reshape(ref[n].shape)
        assert np.array_equal(g, ref[n]), n
    if c.od["kind"] == orc.DYNAMIC_TOPK:
        bits = orc.keep_bits(c.od["key_bias"], c.od["topk"])
        g = c.lists.tensors["keep_bits"].cpu().numpy().view(np.uint32).reshape(bits.shape)
        assert np.array_equal(g, bits)
        if "keep_idx" in c.lists.tensors:
            idx = orc.keep_index(c.od["key_bias"], c.od["topk"])
            g = c.lists.tensors["keep_idx"].cpu().numpy().reshape(idx.shape)
            assert np.array_equal(g, idx)


# ------------------------------------------------------------------ a1 build_block_mask
@pytest.mark.parametrize("kind", ["causal", "sliding", "block_diag", "prefix_lm", "dynamic", "none", "mini_causal"])
@pytest.mark.parametrize("Sq,Sk,sm,sn", [(1000, 1000, 256, 512), (383, 769, 256, 256), (1025, 511, 128, 128),
                                         (640, 512, 256, 512), (129, 257, 128, 256)])
def test_block_mask_bit_exact(kind, Sq, Sk, sm, sn):
    c = Case(1, 2, Sq, Sk, 64, 64, kind, sparse=(sm, sn), prefix_len=100, block_size=192)
    torch.cuda.synchronize()
    lists_equal(c, 1, 2, Sq, Sk, sm, sn)
    assert_no_device_error()


# more than 256 sparse blocks along a list: the list builder compacts each
# row / column in chunks of 256 blocks, so the entries cross a chunk boundary
@pytest.mark.parametrize("kind", ["causal", "sliding", "prefix_lm", "none"])
@pytest.mark.parametrize("Sq,Sk", [(300, 33000), (33000, 300)])
def test_block_mask_bit_exact_past_256_blocks(kind, Sq, Sk):
    c = Case(1, 1, Sq, Sk, 64, 64, kind, sparse=(128, 128), prefix_len=20000, window=17000)
    torch.cuda.synchronize()
    lists_equal(c, 1, 1, Sq, Sk, 128, 128)
    assert_no_device_error()


@pytest.mark.parametrize("topk", [0, 1, 33, 699, 700, 5000])
def test_keep_index_bit_exact(topk):
    c = Case(2, 2, 64, 700, 64, 64, "dynamic", topk=topk, sparse=(128, 128))
    torch.cuda.synchronize()
    lists_equal(c, 2, 2, 64, 700, 128, 128)


def test_topk_ties_and_signed_zeros():
    B, H, Sk = 1, 3, 700
    c = Case(B, H, 64, Sk, 64, 64, "dynamic", topk=100)
    kb = torch.randn(B, H, Sk, generator=torch.Generator().manual_seed(5))
    kb = torch.round(kb * 2) / 2  # many ties
    kb[0, 1, :50] = 0.0
    kb[0, 1, 50:100] = -0.0
    kb[0, 2] = 1.0  # all equal: lowest indices win
    c.dev["key_bias"].copy_(kb)
    c.od["key_bias"] = kb.double().numpy()
    ga.build_block_mask(B, H, 64, Sk, c.spec, c.lists)
    torch.cuda.synchronize()
    lists_equal(c, B, H, 64, Sk, 256, 512)


# ------------------------------------------------------------------ a2 forward (bf16, tensor cores)
FWD_CASES = [
    # B, H, Sq, Sk, Dqk, Dv, kind, extras
    (1, 2, 300, 300, 64, 64, "none", {}),
    (1, 2, 1000, 1000, 64, 64, "causal", {}),
    (2, 1, 640, 700, 128, 128, "causal", dict(slope=0.01)),
    (1, 2, 513, 769, 192, 128, "sliding", dict(slope=0.01)),
    (1, 1, 1024, 1024, 192, 128, "block_diag", dict(block_size=256)),
    (1, 2, 700, 700, 32, 32, "prefix_lm", dict(prefix_len=300)),
    (1, 2, 900, 900, 64, 64, "dynamic", dict(topk=200)),
    (1, 1, 256, 384, 128, 128, "causal", dict(softcap=2.0, use_bias=True)),
    (1, 1, 1025, 511, 128, 128, "sliding", {}),
    (1, 2, 1000, 1000, 64, 64, "mini_causal", dict(block_size=192)),
    (1, 1, 513, 769, 192, 128, "mini_causal", dict(block_size=128, slope=0.01)),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: f"{c[6]}-{c[2]}x{c[3]}-d{c[4]}")
def test_forward_bf16(case):
    B, H, Sq, Sk, Dqk, Dv, kind, ex = case
    c = Case(B, H, Sq, Sk, Dqk, Dv, kind, **ex)
    o, lse = c.fwd()
    torch.cuda.synchronize()
    assert_no_device_error()
    for b in range(B):
        for h in range(H):
            o_ref, l_ref = c.problem(b, h).forward()
            check_out(f64(o[b, h]), o_ref)
            check_lse(f64(lse[b, h]), l_ref)


@pytest.mark.parametrize("row", read_golden("fa_pr2661_fuzz_cases.txt"), ids=lambda r: r[0])
def test_forward_fuzz_shapes(row):
    seed, sq, sk, dqk, dv, stm, stn, name = row
    c = Case(1, 1, int(sq), int(sk), int(dqk), int(dv), name, seed=int(seed), sparse=(int(stm), int(stn)),
             slope=0.01, block_size=256)
    o, lse = c.fwd()
    torch.cuda.synchronize()
    o_ref, l_ref = c.problem(0, 0).forward()
    check_out(f64(o[0, 0]), o_ref)
    check_lse(f64(lse[0, 0]), l_ref)
    assert_no_device_error()


# ------------------------------------------------------------------ a3-a5 backward (bf16)
BWD_CASES = [
    (1, 2, 400, 400, 64, 64, "causal", {}),
    (1, 1, 513, 769, 192, 128, "sliding", dict(slope=0.01)),
    (1, 2, 384, 384, 128, 128, "none", {}),
    (1, 1, 600, 600, 32, 32, "prefix_lm", dict(prefix_len=200)),
    (1, 1, 700, 700, 64, 64, "dynamic", dict(topk=150)),
    (1, 1, 512, 512, 192, 128, "block_diag", dict(block_size=256)),
    (1, 1, 300, 260, 128, 128, "causal", dict(softcap=2.0, use_bias=True)),
    (1, 2, 700, 640, 64, 64, "mini_causal", dict(block_size=200)),
]


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"{c[6]}-{c[2]}x{c[3]}-d{c[4]}")
def test_backward_bf16(case, deterministic):
    B, H, Sq, Sk, Dqk, Dv, kind, ex = case
    c = Case(B, H, Sq, Sk, Dqk, Dv, kind, **ex)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse, deterministic)
    torch.cuda.synchronize()
    assert_no_device_error()
    for b in range(B):
        for h in range(H):
            dq_r, dk_r, dv_r, _ = c.problem(b, h).backward(c.h["do"][b, h])
            check_grad(f64(dq[b, h]), dq_r, "dQ")
            check_grad(f64(dk[b, h]), dk_r, "dK")
            check_grad(f64(dv[b, h]), dv_r, "dV")


def test_gradients_are_bitwise_reproducible():
    # no atomics anywhere in the backward: repeated runs, and either value of
    # the deterministic flag, give identical bits
    c = Case(1, 2, 640, 640, 128, 128, "causal")
    o, lse = c.fwd()
    a = c.bwd(o, lse, True)
    b = c.bwd(o, lse, True)
    d = c.bwd(o, lse, False)
    torch.cuda.synchronize()
    for x, y, z in zip(a, b, d):
        assert torch.equal(x, y) and torch.equal(x, z)


# ------------------------------------------------------------------ gathered dynamic path + key-bias gradient
GATHER_CASES = [
    # B, H, Sq, Sk, D, topk, extras
    (1, 2, 900, 900, 64, 200, {}),
    (1, 2, 1000, 1000, 32, 300, {}),
    (2, 1, 700, 1000, 128, 300, dict(slope=0.01)),        # Sq < Sk
    (1, 1, 1000, 700, 64, 650, {}),                       # Sq > Sk: leading rows see few keys
    (1, 1, 640, 640, 64, 1, {}),                          # one kept key
    (1, 1, 513, 513, 64, 600, {}),                        # topk >= Sk: every key kept
    (1, 1, 777, 777, 128, 260, dict(softcap=2.0, slope=0.02)),
    (1, 1, 640, 900, 192, 333, dict(slope=0.01)),         # MLA head dims
]


@pytest.mark.parametrize("gather", [True, False])
@pytest.mark.parametrize("case", GATHER_CASES, ids=lambda c: f"{c[2]}x{c[3]}-d{c[4]}-k{c[5]}")
def test_dynamic_forward_backward_dkey_bias(case, gather):
    # gather=True streams only the kept keys (compact tiles); gather=False
    # walks the block lists and tests the keep bits: both against the oracle
    B, H, Sq, Sk, D, topk, ex = case
    Dv = 128 if D == 192 else D
    c = Case(B, H, Sq, Sk, D, Dv, "dynamic", topk=topk, sparse=(128, 128), gather=gather, **ex)
    o, lse = c.fwd()
    db = c.dbias_buffer()
    dq, dk, dv = c.bwd(o, lse, dkey_bias=db)
    torch.cuda.synchronize()
    assert_no_device_error()
    for b in range(B):
        for h in range(H):
            p = c.problem(b, h)
            o_ref, l_ref = p.forward()
            check_out(f64(o[b, h]), o_ref)
            check_lse(f64(lse[b, h]), l_ref)
            dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][b, h])
            check_grad(f64(dq[b, h]), dq_r, "dQ")
            check_grad(f64(dk[b, h]), dk_r, "dK")
            check_grad(f64(dv[b, h]), dv_r, "dV")
            check_dbias(f64(db[b, h]), p.dkey_bias(c.h["do"][b, h]))
            # keys outside the keep set get exactly zero gradients
            keep = orc.topk_keep(c.od["key_bias"][b, h], topk)
            assert np.all(f64(dk[b, h])[~keep] == 0) and np.all(f64(dv[b, h])[~keep] == 0)
            assert np.all(f64(db[b, h])[~keep] == 0)


@pytest.mark.parametrize("case", [(1, 2, 600, 600, 64, "causal", {}),
                                  (1, 1, 513, 769, 192, "sliding", dict(slope=0.01)),
                                  (1, 1, 384, 384, 128, "none", dict(softcap=2.0)),
                                  (1, 1, 600, 600, 32, "prefix_lm", dict(prefix_len=200)),
                                  (1, 1, 512, 512, 64, "block_diag", dict(block_size=128))],
                         ids=lambda c: c[5])
def test_key_bias_gradient_bf16(case):
    B, H, Sq, Sk, D, kind, ex = case
    Dv = 128 if D == 192 else D
    c = Case(B, H, Sq, Sk, D, Dv, kind, use_bias=True, sparse=(128, 256), **ex)
    o, lse = c.fwd()
    db = c.dbias_buffer()
    c.bwd(o, lse, dkey_bias=db)
    torch.cuda.synchronize()
    assert_no_device_error()
    for h in range(H):
        check_dbias(f64(db[0, h]), c.problem(0, h).dkey_bias(c.h["do"][0, h]))


def test_gathered_gradients_are_bitwise_reproducible():
    c = Case(1, 2, 900, 900, 64, 64, "dynamic", topk=300, sparse=(128, 128))
    o, lse = c.fwd()
    d1, d2 = c.dbias_buffer(), c.dbias_buffer()
    a = c.bwd(o, lse, dkey_bias=d1)
    b = c.bwd(o, lse, dkey_bias=d2)
    torch.cuda.synchronize()
    for x, y in zip(a + (d1,), b + (d2,)):
        assert torch.equal(x, y)


# ------------------------------------------------------------------ grouped-query attention (GQA)
GQA_CASES = [
    # B, H, Hkv, Sq, Sk, Dqk, Dv, kind, extras, dtype
    (1, 4, 2, 640, 700, 128, 128, "causal", dict(slope=0.01), "bf16"),
    (2, 8, 1, 513, 513, 64, 64, "sliding", {}, "bf16"),
    (1, 6, 2, 512, 640, 192, 128, "block_diag", dict(block_size=256), "bf16"),
    (1, 4, 2, 700, 700, 64, 64, "dynamic", dict(topk=250), "bf16"),       # per-head keep sets, shared K/V
    (1, 4, 1, 384, 300, 32, 32, "prefix_lm", dict(prefix_len=100, softcap=2.0, use_bias=True), "bf16"),
    (1, 4, 2, 150, 170, 32, 16, "causal", dict(slope=0.02), "fp32"),
]


@pytest.mark.parametrize("case", GQA_CASES, ids=lambda c: f"{c[7]}-h{c[1]}kv{c[2]}-{c[9]}")
def test_gqa_forward_backward(case):
    # dK / dV of a key/value head are the sums over its query heads
    B, H, Hkv, Sq, Sk, Dqk, Dv, kind, ex, dt = case
    c = Case(B, H, Sq, Sk, Dqk, Dv, kind, dtype=dt, Hkv=Hkv, sparse=(128, 256), **ex)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    assert dk.shape == (B, Hkv, Sk, Dqk) and dv.shape == (B, Hkv, Sk, Dv)
    fp32 = dt == "fp32"
    G = H // Hkv
    for b in range(B):
        for hk in range(Hkv):
            dk_r = np.zeros((Sk, Dqk))
            dv_r = np.zeros((Sk, Dv))
            for h in range(hk * G, (hk + 1) * G):
                p = c.problem(b, h)
                o_ref, l_ref = p.forward()
                check_out(f64(o[b, h]), o_ref, fp32=fp32)
                check_lse(f64(lse[b, h]), l_ref, fp32=fp32)
                dq_r, dkh, dvh, _ = p.backward(c.h["do"][b, h])
                check_grad(f64(dq[b, h]), dq_r, "dQ", fp32=fp32)
                dk_r += dkh
                dv_r += dvh
            check_grad(f64(dk[b, hk]), dk_r, "dK", fp32=fp32)
            check_grad(f64(dv[b, hk]), dv_r, "dV", fp32=fp32)


@pytest.mark.parametrize("n", [1, 4])
@pytest.mark.parametrize("H,Hkv,Sq,D,kind", [(4, 2, 2, 128, "causal"),    # 4 rows per group: 1 row per lane group
                                             (4, 1, 2, 128, "causal"),    # 8 rows
                                             (16, 2, 3, 128, "causal"),   # 24 rows: two CTAs of 16 rows
                                             (8, 1, 1, 64, "none"),       # MQA-style, D=64
                                             (6, 3, 1, 128, "none"),      # 2 rows per group
                                             (64, 1, 3, 128, "causal")])  # 192 rows: two 128-row tiles
def test_gqa_splitkv_decode(n, H, Hkv, Sq, D, kind):
    c = Case(2, H, Sq, 1500, D, D, kind, Hkv=Hkv, lists=False, sparse=None)
    o, lse = ga.attn_fwd_splitkv(c.dev["q"], c.dev["k"], c.dev["v"], 0.0, c.spec, n)
    torch.cuda.synchronize()
    assert_no_device_error()
    for b in range(2):
        for h in range(H):
            o_ref, l_ref = c.problem(b, h).forward()
            check_out(f64(o[b, h]), o_ref)
            check_lse(f64(lse[b, h]), l_ref)


def _paged_cache(k, v, page_size, seqlens, extra_pages, seed):
    """Scatter dense per-sequence K/V [B, Hkv, S, D] into a shuffled page pool
    [num_pages, Hkv, page_size, D] and its page table (test set-up only)."""
    B, Hkv, S, D = k.shape
    need = [-(-int(n) // page_size) for n in seqlens]
    max_pages = max(1, max(need))
    num_pages = sum(need) + extra_pages
    rng = np.random.default_rng(seed)
    order = rng.permutation(num_pages)
    kc = torch.zeros(num_pages, Hkv, page_size, D, dtype=k.dtype)
    vc = torch.zeros_like(kc)
    table = np.full((B, max_pages), 10 ** 6, dtype=np.int32)  # unused entries: never read
    t = 0
    for b in range(B):
        for pgi in range(need[b]):
            pg = int(order[t])
            t += 1
            table[b, pgi] = pg
            r0, r1 = pgi * page_size, min((pgi + 1) * page_size, int(seqlens[b]))
            kc[pg, :, : r1 - r0] = k[b, :, r0:r1]
            vc[pg, :, : r1 - r0] = v[b, :, r0:r1]
    return kc, vc, torch.from_numpy(table)


@pytest.mark.parametrize("page_size,n,kind,Hkv,H", [(64, 1, "none", 2, 4), (128, 4, "causal", 1, 4),
                                                     (256, 16, "none", 4, 4), (192, 2, "causal", 2, 4),
                                                     (128, 2, "causal", 1, 16), (256, 1, "none", 2, 8)])
def test_paged_splitkv_decode(page_size, n, kind, Hkv, H):
    B, Sq, S, D = 4, 2, 1100, 128
    c = Case(B, H, Sq, S, D, D, kind, Hkv=Hkv, lists=False, sparse=None)
    seqlens = np.array([1100, 0, 1, 777])
    kc, vc, table = _paged_cache(c.x["k"], c.x["v"], page_size, seqlens, extra_pages=3, seed=page_size)
    o, lse = ga.attn_fwd_splitkv_paged(c.dev["q"], kc.cuda(), vc.cuda(), table.cuda(),
                                       torch.from_numpy(seqlens.astype(np.int32)).cuda(), 0.0, c.spec, n)
    torch.cuda.synchronize()
    assert_no_device_error()
    G = H // Hkv
    for b in range(B):
        L = int(seqlens[b])
        for h in range(H):
            if L == 0:
                assert np.all(f64(o[b, h]) == 0) and np.all(np.isneginf(f64(lse[b, h])))
                continue
            p = orc.Problem(c.h["q"][b, h], c.h["k"][b, h // G][:L], c.h["v"][b, h // G][:L], kind=c.od["kind"])
            o_ref, l_ref = p.forward()
            check_out(f64(o[b, h]), o_ref)
            check_lse(f64(lse[b, h]), l_ref)


@pytest.mark.parametrize("H,Hkv,page", [(2, 2, 64), (4, 1, 128)])  # per-row kernel; packed tensor-core path
def test_paged_decode_bad_page_index_raises_device_error(H, Hkv, page):
    # a page index outside the pool is not read: the kernel flags it
    B, D = 1, 64
    q = torch.randn(B, H, 1, D).to(torch.bfloat16).cuda()
    kc = torch.zeros(2, Hkv, page, D, dtype=torch.bfloat16).cuda()
    table = torch.tensor([[0, 5]], dtype=torch.int32).cuda()
    seqlens = torch.tensor([page + 36], dtype=torch.int32).cuda()
    ga.attn_fwd_splitkv_paged(q, kc, kc, table, seqlens, 0.0, None, 1)
    torch.cuda.synchronize()
    assert ga.load_library().gbattn_last_device_error(None) == ga.binding.ERR_BLOCKS


# ------------------------------------------------------------------ element-table masks (arbitrary predicates)
@pytest.mark.parametrize("pattern,per_head,Sq,Sk,sm,sn", [("random", False, 700, 900, 128, 128),
                                                          ("documents", True, 1000, 1000, 256, 512),
                                                          ("dilated", False, 513, 769, 128, 256)])
def test_table_block_lists_bit_exact(pattern, per_head, Sq, Sk, sm, sn):
    t = make_table(1, 2, Sq, Sk, pattern, per_head)
    c = Case(1, 2, Sq, Sk, 64, 64, "table", table=t, sparse=(sm, sn))
    torch.cuda.synchronize()
    lists_equal(c, 1, 2, Sq, Sk, sm, sn)
    assert_no_device_error()


TABLE_CASES = [
    # B, H, Hkv, Sq, Sk, Dqk, Dv, pattern, per_head, sparse, extras, dtype
    (1, 2, 2, 700, 900, 64, 64, "random", False, (128, 128), {}, "bf16"),
    (1, 2, 2, 1000, 1000, 128, 128, "documents", True, (256, 512), dict(slope=0.01), "bf16"),
    (1, 2, 2, 513, 769, 192, 128, "dilated", False, (128, 256), dict(softcap=2.0, use_bias=True), "bf16"),
    (1, 4, 2, 640, 640, 64, 64, "random", True, (128, 128), {}, "bf16"),       # GQA with per-head tables
    (1, 2, 2, 150, 170, 32, 16, "documents", True, (128, 128), {}, "fp32"),
]


@pytest.mark.parametrize("case", TABLE_CASES, ids=lambda c: f"{c[7]}-{'head' if c[8] else 'shared'}-d{c[5]}-{c[11]}")
def test_table_forward_backward(case):
    B, H, Hkv, Sq, Sk, Dqk, Dv, pattern, per_head, sparse, ex, dt = case
    t = make_table(B, H, Sq, Sk, pattern, per_head)
    c = Case(B, H, Sq, Sk, Dqk, Dv, "table", dtype=dt, Hkv=Hkv, table=t, sparse=sparse, **ex)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    fp32 = dt == "fp32"
    G = H // Hkv
    for b in range(B):
        for hk in range(Hkv):
            dk_r, dv_r = 0.0, 0.0
            for h in range(hk * G, (hk + 1) * G):
                p = c.problem(b, h)
                o_ref, l_ref = p.forward()
                check_out(f64(o[b, h]), o_ref, fp32=fp32)
                check_lse(f64(lse[b, h]), l_ref, fp32=fp32)
                dq_r, dkh, dvh, _ = p.backward(c.h["do"][b, h])
                check_grad(f64(dq[b, h]), dq_r, "dQ", fp32=fp32)
                dk_r = dk_r + dkh
                dv_r = dv_r + dvh
            check_grad(f64(dk[b, hk]), dk_r, "dK", fp32=fp32)
            check_grad(f64(dv[b, hk]), dv_r, "dV", fp32=fp32)


# ------------------------------------------------------------------ fp32 path
@pytest.mark.parametrize("case", [(1, 1, 128, 128, 64, 64, "causal", {}),
                                  (1, 2, 200, 333, 48, 24, "sliding", dict(window=50, slope=0.02)),
                                  (1, 1, 150, 150, 64, 64, "dynamic", dict(topk=40)),
                                  (1, 1, 130, 100, 16, 16, "block_diag", dict(block_size=64, softcap=1.5)),
                                  (1, 1, 150, 130, 32, 32, "mini_causal", dict(block_size=48))],
                         ids=lambda c: c[6])
def test_fp32_forward_backward(case):
    B, H, Sq, Sk, Dqk, Dv, kind, ex = case
    c = Case(B, H, Sq, Sk, Dqk, Dv, kind, dtype="fp32", sparse=(128, 128), **ex)
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    assert_no_device_error()
    for h in range(H):
        p = c.problem(0, h)
        o_ref, l_ref = p.forward()
        check_out(f64(o[0, h]), o_ref, fp32=True)
        check_lse(f64(lse[0, h]), l_ref, fp32=True)
        dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, h])
        check_grad(f64(dq[0, h]), dq_r, "dQ", fp32=True)
        check_grad(f64(dk[0, h]), dk_r, "dK", fp32=True)
        check_grad(f64(dv[0, h]), dv_r, "dV", fp32=True)


@pytest.mark.parametrize("kind,ex", [("dynamic", dict(topk=40)), ("causal", dict(softcap=1.5, slope=0.02))])
def test_fp32_key_bias_gradient(kind, ex):
    c = Case(1, 2, 150, 170, 32, 16, kind, dtype="fp32", use_bias=True, sparse=(128, 128), **ex)
    o, lse = c.fwd()
    db = c.dbias_buffer()
    c.bwd(o, lse, dkey_bias=db)
    torch.cuda.synchronize()
    for h in range(2):
        check_dbias(f64(db[0, h]), c.problem(0, h).dkey_bias(c.h["do"][0, h]), fp32=True)


# ------------------------------------------------------------------ a6-a7 split-KV decode
# split counts of the [FSA] test set-up (tests/golden/fsa_pr148_test_setup.txt)
@pytest.mark.parametrize("n", golden_setup()["splits"])
@pytest.mark.parametrize("D,Sq,Sk,kind", [(128, 1, 3000, "none"), (64, 3, 1100, "causal"), (128, 2, 77, "none")])
def test_splitkv_decode(n, D, Sq, Sk, kind):
    c = Case(2, 3, Sq, Sk, D, D, kind, lists=False, sparse=None)
    o, lse = ga.attn_fwd_splitkv(c.dev["q"], c.dev["k"], c.dev["v"], 0.0, c.spec, n)
    torch.cuda.synchronize()
    assert_no_device_error()
    for b in range(2):
        for h in range(3):
            o_ref, l_ref = c.problem(b, h).forward()
            check_out(f64(o[b, h]), o_ref)
            check_lse(f64(lse[b, h]), l_ref)


# ------------------------------------------------------------------ edge cases
def test_fully_masked_rows_and_empty_lists():
    # block-diagonal with Sq > Sk: the first Sq - Sk rows see no key at all
    c = Case(1, 1, 400, 150, 64, 64, "block_diag", block_size=64, sparse=(128, 128))
    o, lse = c.fwd()
    dq, dk, dv = c.bwd(o, lse)
    torch.cuda.synchronize()
    p = c.problem(0, 0)
    o_ref, l_ref = p.forward()
    check_out(f64(o[0, 0]), o_ref)
    check_lse(f64(lse[0, 0]), l_ref)
    assert np.all(f64(o[0, 0])[:250] == 0.0)
    dq_r, dk_r, dv_r, _ = p.backward(c.h["do"][0, 0])
    assert np.all(f64(dq[0, 0])[:250] == 0.0)
    check_grad(f64(dk[0, 0]), dk_r, "dK")
    check_grad(f64(dv[0, 0]), dv_r, "dV")


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (1, 300), (300, 1), (129, 1)])
def test_tiny_and_single_key_shapes(Sq, Sk):
    c = Case(1, 2, Sq, Sk, 64, 64, "none", lists=False, sparse=None)
    o, lse = c.fwd()
    torch.cuda.synchronize()
    for h in range(2):
        o_ref, l_ref = c.problem(0, h).forward()
        check_out(f64(o[0, h]), o_ref)
        check_lse(f64(lse[0, h]), l_ref)
