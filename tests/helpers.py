"""Shared test helpers: run one case through the C ABI and through the oracle
on the same seeded inputs, and compare with the stated tolerances.

Tolerances (bf16): O elementwise |g - r| <= 2e-2 + 2e-2 |r|; LSE |g - r| <=
2e-2 (-inf must match); dQ/dK/dV max|g - r| / max|r| <= 5e-2. fp32 path:
atol = rtol = 1e-4 (the fp32 tolerance of the POPCORNBENCH "Kimi-K2.6
l1_p97" SDPA task).
"""
import numpy as np
import torch

import block_sparse_attention_tma_gb300 as ga
from block_sparse_attention_tma_gb300.synth import make_inputs
from oracle import attention as orc

KIND = {"none": orc.NONE, "causal": orc.CAUSAL, "sliding": orc.SLIDING, "sliding_window": orc.SLIDING,
        "block_diag": orc.BLOCK_DIAG, "block_diagonal": orc.BLOCK_DIAG, "prefix_lm": orc.PREFIX_LM,
        "dynamic": orc.DYNAMIC_TOPK, "mini_causal": orc.MINI_CAUSAL, "table": orc.TABLE}


def spec_dicts(kind, Sq, Sk, window=None, block_size=256, prefix_len=64, topk=None, slope=0.0, softcap=0.0,
               key_bias=None):
    k = KIND[kind]
    d = dict(kind=k, rel_bias_slope=slope, softcap=softcap)
    if k == orc.SLIDING:
        d["window_left"] = max(64, min(Sq, Sk) // 3) if window is None else window
    if k in (orc.BLOCK_DIAG, orc.MINI_CAUSAL):
        d["block_size"] = block_size
    if k == orc.PREFIX_LM:
        d["prefix_len"] = prefix_len
    if k == orc.DYNAMIC_TOPK:
        d["topk"] = max(1, Sk // 4) if topk is None else topk
    return d


def to_gpu_spec(d, key_bias_gpu=None, table_gpu=None):
    return ga.MaskSpec(kind=d["kind"], window_left=d.get("window_left", -1), block_size=d.get("block_size", 0),
                       prefix_len=d.get("prefix_len", 0), topk=d.get("topk", 0),
                       rel_bias_slope=d.get("rel_bias_slope", 0.0), softcap=d.get("softcap", 0.0),
                       key_bias=key_bias_gpu, table=table_gpu)


def make_table(B, H, Sq, Sk, pattern="random", per_head=False, seed=7):
    """A boolean element table for the TABLE kind (test set-up): "random"
    (35% of pairs), "dilated" (causal, every other key), or "documents"
    (causal inside documents of random lengths)."""
    rng = np.random.default_rng(seed)
    shape = (B, H, Sq, Sk) if per_head else (Sq, Sk)
    i = np.arange(Sq)[:, None] + (Sk - Sq)
    j = np.arange(Sk)[None, :]
    if pattern == "random":
        return rng.random(shape) < 0.35
    if pattern == "dilated":
        t = (j <= i) & ((i - j) % 2 == 0)
    elif pattern == "documents":
        cuts = np.sort(rng.choice(np.arange(1, Sk), size=min(6, Sk - 1), replace=False))
        doc = np.searchsorted(cuts, np.arange(Sk), side="right")
        t = (j <= i) & (doc[np.clip(i, 0, Sk - 1)] == doc[j[0]][None, :])
    else:
        raise ValueError(pattern)
    return np.broadcast_to(t, shape).copy()


def f64(t):
    return t.detach().float().cpu().double().numpy()


class Case:
    """Inputs on host and device, the GPU spec and lists, and the oracle spec."""

    def __init__(self, B, H, Sq, Sk, Dqk, Dv, kind="none", dtype="bf16", seed=42, sparse=(256, 512),
                 use_bias=False, lists=True, gather=True, Hkv=None, table=None, **kw):
        need_bias = use_bias or KIND[kind] == orc.DYNAMIC_TOPK
        self.shape = (B, H, Sq, Sk, Dqk, Dv)
        self.Hkv = H if Hkv is None else Hkv
        self.G = H // self.Hkv
        self.x = make_inputs(B, H, Sq, Sk, Dqk, Dv, dtype, seed=seed, bias=need_bias, Hkv=self.Hkv)
        self.dev = {n: t.cuda() for n, t in self.x.items()}
        self.d = spec_dicts(kind, Sq, Sk, **kw)
        self.table = table
        tab_gpu = None
        if table is not None:
            tab_gpu = ga.pack_mask_table(torch.from_numpy(np.ascontiguousarray(table)).cuda())
            self.dev["table"] = tab_gpu
        self.spec = to_gpu_spec(self.d, self.dev.get("key_bias"), tab_gpu)
        self.lists = None
        if lists and (self.d["kind"] != orc.NONE or sparse is not None):
            sm, sn = sparse
            self.lists = ga.alloc_block_lists(B, H, Sq, Sk, sm, sn, gather=gather)
            ga.build_block_mask(B, H, Sq, Sk, self.spec, self.lists)
        od = dict(self.d)
        if table is not None:
            od["table"] = table
        if need_bias:
            od["key_bias"] = self.x["key_bias"].double().numpy()
        self.od = od
        self.h = {n: f64(t) for n, t in self.x.items() if n != "key_bias"}

    def fwd(self):
        return ga.attn_fwd(self.dev["q"], self.dev["k"], self.dev["v"], 0.0, self.spec, self.lists)

    def bwd(self, o, lse, deterministic=False, dkey_bias=None):
        return ga.attn_bwd(self.dev["q"], self.dev["k"], self.dev["v"], o, self.dev["do"], lse, 0.0, self.spec,
                           self.lists, deterministic=deterministic, dkey_bias=dkey_bias)

    def dbias_buffer(self):
        B, H, Sq, Sk = self.shape[:4]
        # filled with NaN so that a key the kernels skip shows up
        return torch.full((B, H, Sk), float("nan"), dtype=torch.float32, device="cuda")

    def problem(self, b, h):
        """Oracle problem of query head h (it reads key/value head h // G)."""
        kb = self.od.get("key_bias")
        hk = h // self.G
        return orc.Problem(self.h["q"][b, h], self.h["k"][b, hk], self.h["v"][b, hk], kind=self.od["kind"],
                           window_left=self.od.get("window_left", -1), block_size=self.od.get("block_size", 0),
                           prefix_len=self.od.get("prefix_len", 0), topk=self.od.get("topk", 0),
                           rel_bias_slope=self.od.get("rel_bias_slope", 0.0), softcap=self.od.get("softcap", 0.0),
                           key_bias=None if kb is None else kb[b, h],
                           table=None if self.table is None else (self.table if self.table.ndim == 2
                                                                  else self.table[b, h]))


def check_out(og, o_ref, fp32=False):
    """bf16: |g - r| <= 2e-2 + 2e-2 |r| elementwise (the absolute and relative
    bound of the task), and, per output row, max |g - r| <= 2e-2 max |r| +
    2e-3: the relative bound taken against the row's scale, which is what
    catches a wrong row whose values are all small (decode rows over many
    keys are ~0.02 in magnitude, inside the absolute bound whatever they are).
    The 2e-3 floor is ~10 bf16 ulps of such a row."""
    if fp32:
        assert np.allclose(og, o_ref, rtol=1e-4, atol=1e-4), np.max(np.abs(og - o_ref))
    else:
        bad = np.abs(og - o_ref) > 2e-2 + 2e-2 * np.abs(o_ref)
        assert not bad.any(), f"O mismatch: {bad.sum()} elements, max abs {np.max(np.abs(og - o_ref)):.3e}"
        if og.ndim >= 1 and og.size:
            err = np.max(np.abs(og - o_ref), axis=-1)
            scale = np.max(np.abs(o_ref), axis=-1)
            rows = err > 2e-2 * scale + 2e-3
            assert not rows.any(), (f"O rows off their own scale: {int(rows.sum())} rows, worst err/scale "
                                    f"{float(np.max(err / np.maximum(scale, 1e-30))):.3e}")


def check_lse(lg, l_ref, fp32=False):
    inf_r = np.isinf(l_ref)
    assert np.array_equal(np.isinf(lg) & (lg < 0), inf_r), "-inf rows differ"
    if (~inf_r).any():
        err = np.max(np.abs(lg[~inf_r] - l_ref[~inf_r]))
        assert err <= (1e-4 if fp32 else 2e-2), f"LSE err {err:.3e}"


def check_dbias(g, r, fp32=False):
    """Key-bias gradient: same bar as dQ/dK/dV (relative to max), and no NaN
    (every key is written)."""
    assert np.all(np.isfinite(g)), "dkey_bias has unwritten (NaN) entries"
    return check_grad(g, r, "dkey_bias", fp32=fp32)


def check_grad(g, r, name, fp32=False):
    if fp32:
        assert np.allclose(g, r, rtol=1e-4, atol=1e-4), f"{name}: {np.max(np.abs(g - r)):.3e}"
        return 0.0
    den = np.max(np.abs(r))
    err = np.max(np.abs(g - r)) / den if den > 0 else np.max(np.abs(g))
    assert err <= 5e-2, f"{name} rel-to-max err {err:.3e}"
    return err


def assert_no_device_error():
    assert ga.load_library().gbattn_last_device_error(None) == 0
