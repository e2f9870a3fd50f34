"""fp64 CPU oracle for masked, block-sparse scaled-dot-product attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (the CUDA library and its Python binding) never
calls it, and this module imports nothing from the product package.

Everything here is the plain definition of the result, written out in float64
with numpy. Scores are materialised, masked, normalised by a two-pass softmax,
multiplied by V. Gradients are the analytic derivative of that definition.
Each output row (forward, dQ) or key column (dK, dV) is defined on its own, so
the functions accept an optional subset of rows/columns to evaluate; nothing
is blocked, fused or reordered beyond that.

Sources (titles of the pages the method is taken from):
  [FSA]  "Optimize Flash Dynamic Mask Attention Kernel Configurations"
         (flash-sparse-attention PR #148): split-KV forward, deterministic
         backward, masks/softcap semantics unchanged vs an SDPA reference.
  [FA2C] "Enable 2CTA for SM100 block-sparse backward" (flash-attention
         PR #2661): block-sparse fwd/bwd lists built from a mask predicate at
         sparse tiles that are multiples of the kernel tile; mask kinds
         causal / sliding_window / block_diagonal / prefix_lm; window rule
         max(64, min(Sq, Sk)//3); score_mod rel_bias whose backward passes the
         gradient through; softmax_scale = 1/sqrt(headdim); reference =
         flex_attention + autograd.
  [PCB]  POPCORNBENCH trace "Kimi-K2.6 l1_p97" (fp32 SDPA kernel): online
         softmax merge algebra (m_new = max(m1, m2); l and o rescaled by
         exp(m - m_new)); fp32 tolerance atol = rtol = 1e-4.

Readings where the pages are silent:
  * Sq != Sk aligns the causal diagonal bottom-right: delta = Sk - Sq.
  * sliding window keeps keys j with 0 <= (i + delta) - j <= window_left
    (window_left + 1 keys, self included); window_left < 0 = unbounded.
  * block_diagonal is bidirectional inside a block of the given size.
  * mini_causal ([FA2C] lists it among the fuzz tester's mask names without
    defining it) is causal inside each block of the given size: the
    block-diagonal mask AND the causal mask.
  * table: an arbitrary element predicate given as a boolean matrix
    [Sq, Sk] (the stand-in for flex_attention's mask_mod, from which [FA2C]
    builds its block lists).
  * prefix_lm allows j < prefix_len or the causal keys.
  * dynamic_topk: per (b, h), keep the first k keys in the order
    (key_bias descending, index ascending), AND causal; the bias is also
    added to the score.
  * order of score terms: scale -> softcap -> + rel bias + key bias -> mask.
  * a row with no allowed key has O = 0, LSE = -inf and zero gradients.
  * LSE is the natural log of sum_j exp(s_ij), biases included.
"""
from __future__ import annotations

import math

import numpy as np

# Mask kinds (numbering is the C ABI's; the oracle keeps its own copy).
NONE, CAUSAL, SLIDING, BLOCK_DIAG, PREFIX_LM, DYNAMIC_TOPK, MINI_CAUSAL, TABLE = range(8)


def default_scale(dqk: int) -> float:
    """softmax_scale = 1/sqrt(headdim) of the QK head dim ([FA2C], fuzz tester
    `run_case`, the `_flash_attn_fwd` call)."""
    return 1.0 / math.sqrt(dqk)


def topk_keep(bias_row: np.ndarray, k: int) -> np.ndarray:
    """Keep-set of the dynamic mask for one (b, h).

    [FSA] title ("Flash Dynamic Mask Attention") names a bias-ranked dynamic
    mask without defining it; the reading taken: the first k keys of the order
    (bias descending, index ascending). All keys are kept when k >= Sk.
    A library sort is the step: lexsort's last key is the primary one.
    """
    sk = bias_row.shape[0]
    keep = np.zeros(sk, dtype=bool)
    if k <= 0:
        return keep
    idx = np.arange(sk)
    order = np.lexsort((idx, -bias_row.astype(np.float64)))
    keep[order[: min(k, sk)]] = True
    return keep


def allowed(kind: int, sq: int, sk: int, rows: np.ndarray, cols: np.ndarray, *,
            window_left: int = -1, block_size: int = 0, prefix_len: int = 0,
            keep: np.ndarray | None = None, table: np.ndarray | None = None) -> np.ndarray:
    """Element mask m_ij (True = the pair (i, j) takes part), rows x cols.

    Mask names follow [FA2C] (`get_mask_pair` names: causal, sliding_window,
    block_diagonal, prefix_lm); the dynamic kind follows [FSA]'s title.
    Positions outside [0, Sq) x [0, Sk) never take part.
    """
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    a = i + (sk - sq)  # bottom-right aligned diagonal
    inb = (i >= 0) & (i < sq) & (j >= 0) & (j < sk)
    if kind == NONE:
        m = np.ones((i.shape[0], j.shape[1]), dtype=bool)
    elif kind == CAUSAL:
        m = j <= a
    elif kind == SLIDING:
        d = a - j
        m = d >= 0
        if window_left >= 0:
            m = m & (d <= window_left)
    elif kind == BLOCK_DIAG:
        if block_size <= 0:
            raise ValueError("block_size must be positive")
        m = np.floor_divide(a, block_size) == np.floor_divide(j, block_size)
    elif kind == PREFIX_LM:
        m = (j < prefix_len) | (j <= a)
    elif kind == TABLE:
        if table is None:
            raise ValueError("table mask needs the element table")
        ii = np.clip(i, 0, sq - 1)
        jj = np.clip(j, 0, sk - 1)
        m = np.asarray(table, dtype=bool)[ii, jj]
    elif kind == MINI_CAUSAL:
        if block_size <= 0:
            raise ValueError("block_size must be positive")
        m = (np.floor_divide(a, block_size) == np.floor_divide(j, block_size)) & (j <= a)
    elif kind == DYNAMIC_TOPK:
        if keep is None:
            raise ValueError("dynamic mask needs the keep set")
        jj = np.clip(j, 0, sk - 1)
        m = keep[jj] & (j <= a)
    else:
        raise ValueError(f"unknown mask kind {kind}")
    return np.broadcast_to(m, (i.shape[0], j.shape[1])) & inb


def _raw_and_scores(q_rows, k, rows, cols, sq, sk, scale, softcap, rel_bias_slope,
                    key_bias_row):
    """r0 = scale * q.k (pre-cap), and s = softcap(r0) + biases.

    Order scale -> softcap -> + biases: flex_attention applies score_mod to the
    scaled score ([FA2C] reference path); the relative bias term is
    slope * (q_idx - kv_idx) ([FA2C] `score_mod_rel_bias`, slope read as 0.01
    in the 16K block-sparse workload); the key bias is added per key.
    """
    r0 = scale * (q_rows @ k[cols].T)
    r = r0
    if softcap > 0.0:
        r = softcap * np.tanh(r0 / softcap)
    s = r
    if rel_bias_slope != 0.0:
        i = np.asarray(rows, dtype=np.float64)[:, None]
        j = np.asarray(cols, dtype=np.float64)[None, :]
        s = s + rel_bias_slope * (i - j)
    if key_bias_row is not None:
        s = s + key_bias_row[cols][None, :]
    return r0, s


def _probs(s, m):
    """Two-pass softmax over allowed entries; fully masked rows -> P = 0,
    LSE = -inf (reading: no key, no output)."""
    sm = np.where(m, s, -np.inf)
    mx = np.max(sm, axis=1, initial=-np.inf)
    live = np.isfinite(mx)
    mx_safe = np.where(live, mx, 0.0)
    e = np.where(m, np.exp(sm - mx_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    lse = np.where(live, mx_safe + np.log(np.where(live, l, 1.0)), -np.inf)
    return p, lse


class Problem:
    """One (b, h) head: float64 copies of what the GPU reads, plus the mask
    parameters. Widening bf16/fp32 to float64 is exact."""

    def __init__(self, q, k, v, *, kind=NONE, scale=None, window_left=-1,
                 block_size=0, prefix_len=0, topk=0, rel_bias_slope=0.0,
                 softcap=0.0, key_bias=None, table=None):
        self.q = np.asarray(q, dtype=np.float64)
        self.k = np.asarray(k, dtype=np.float64)
        self.v = np.asarray(v, dtype=np.float64)
        self.sq, self.dqk = self.q.shape
        self.sk = self.k.shape[0]
        self.dv = self.v.shape[1]
        self.kind = kind
        self.scale = default_scale(self.dqk) if (scale is None or scale <= 0) else float(scale)
        self.window_left = window_left
        self.block_size = block_size
        self.prefix_len = prefix_len
        self.rel_bias_slope = float(rel_bias_slope)
        self.softcap = float(softcap)
        self.key_bias = None if key_bias is None else np.asarray(key_bias, dtype=np.float64)
        self.table = None if table is None else np.asarray(table, dtype=bool)
        self.keep = None
        if kind == DYNAMIC_TOPK:
            if self.key_bias is None:
                raise ValueError("dynamic mask needs a key bias")
            self.keep = topk_keep(self.key_bias, topk)

    def mask(self, rows, cols):
        return allowed(self.kind, self.sq, self.sk, rows, cols,
                       window_left=self.window_left, block_size=self.block_size,
                       prefix_len=self.prefix_len, keep=self.keep, table=self.table)

    def scores(self, rows, cols):
        return _raw_and_scores(self.q[rows], self.k, rows, cols, self.sq, self.sk,
                               self.scale, self.softcap, self.rel_bias_slope,
                               self.key_bias)

    def probs(self, rows):
        """P[rows, :] and LSE[rows] (softmax of the masked scores)."""
        cols = np.arange(self.sk)
        _, s = self.scores(rows, cols)
        return _probs(s, self.mask(rows, cols))

    def forward(self, rows=None, chunk=2048):
        """O[rows] = P[rows] V and LSE[rows] ([PCB] SDPA definition; [FA2C]
        `_flash_attn_fwd(..., return_lse=True)`)."""
        rows = np.arange(self.sq) if rows is None else np.asarray(rows)
        o = np.zeros((rows.shape[0], self.dv))
        lse = np.zeros(rows.shape[0])
        for c0 in range(0, rows.shape[0], chunk):
            rr = rows[c0:c0 + chunk]
            p, l = self.probs(rr)
            o[c0:c0 + chunk] = p @ self.v
            lse[c0:c0 + chunk] = l
        return o, lse

    def backward(self, do, rows=None, cols=None, chunk=2048):
        """Analytic gradients of O = softmax(S) V for L = <dO, O>.

        D_i = sum_d dO_id O_id; dP = dO V^T; dS = P o (dP - D);
        softcap: dS <- dS (1 - tanh^2(r0/c)); dQ = scale dS K;
        dK = scale dS^T Q; dV = P^T dO. Biases are constants (the rel-bias
        score_mod backward returns the incoming gradient, [FA2C]).
        Returns dQ[rows], dK[cols], dV[cols] and D (all rows).
        """
        do = np.asarray(do, dtype=np.float64)
        rows = np.arange(self.sq) if rows is None else np.asarray(rows)
        cols = np.arange(self.sk) if cols is None else np.asarray(cols)
        all_rows = np.arange(self.sq)
        o_all, lse_all = self.forward(all_rows, chunk=chunk)
        d_all = np.sum(do * o_all, axis=1)
        allk = np.arange(self.sk)

        def ds_block(rr, cc):
            p, ds_s, r0 = self._p_ds(do, d_all, lse_all, rr, cc)
            ds = ds_s
            if self.softcap > 0.0:
                t = np.tanh(r0 / self.softcap)
                ds = ds_s * (1.0 - t * t)
            return p, ds

        dq = np.zeros((rows.shape[0], self.dqk))
        for c0 in range(0, rows.shape[0], chunk):
            rr = rows[c0:c0 + chunk]
            _, ds = ds_block(rr, allk)
            dq[c0:c0 + chunk] = self.scale * (ds @ self.k)
        dk = np.zeros((cols.shape[0], self.dqk))
        dv = np.zeros((cols.shape[0], self.dv))
        for c0 in range(0, cols.shape[0], chunk):
            cc = cols[c0:c0 + chunk]
            p, ds = ds_block(all_rows, cc)
            dk[c0:c0 + chunk] = self.scale * (ds.T @ self.q)
            dv[c0:c0 + chunk] = p.T @ do
        return dq, dk, dv, d_all

    def _p_ds(self, do, d_all, lse_all, rr, cc):
        """P and dL/ds (s = the score after the softcap and the biases) on
        rows rr x cols cc, with the raw scaled score r0 for the softcap factor:
        dL/ds_ij = P_ij (dP_ij - D_i)."""
        r0, s = self.scores(rr, cc)
        m = self.mask(rr, cc)
        lse = lse_all[rr]
        live = np.isfinite(lse)
        use = m & live[:, None]
        p = np.exp(np.where(use, s - np.where(live, lse, 0.0)[:, None], -np.inf))
        dp = do[rr] @ self.v[cc].T
        return p, p * (dp - d_all[rr][:, None]), r0

    def dkey_bias(self, do, cols=None, chunk=2048):
        """Gradient of L = <dO, O> with respect to the key bias:
        dL/dkb_j = sum_i dL/ds_ij, because kb_j enters every score s_ij of key
        j with coefficient 1 and is added after the softcap (so the tanh
        factor does not apply). The dynamic keep set is held fixed (it is
        piecewise constant in the bias). Returns dkb[cols]."""
        do = np.asarray(do, dtype=np.float64)
        cols = np.arange(self.sk) if cols is None else np.asarray(cols)
        all_rows = np.arange(self.sq)
        o_all, lse_all = self.forward(all_rows, chunk=chunk)
        d_all = np.sum(do * o_all, axis=1)
        out = np.zeros(cols.shape[0])
        for c0 in range(0, cols.shape[0], chunk):
            cc = cols[c0:c0 + chunk]
            _, ds_s, _ = self._p_ds(do, d_all, lse_all, all_rows, cc)
            out[c0:c0 + chunk] = ds_s.sum(axis=0)
        return out

    # ---- split-KV ([FSA] split-KV forward; [PCB] merge algebra) ----
    @staticmethod
    def split_bounds(sk: int, n: int):
        """Split s covers keys [s*L, min((s+1)*L, Sk)), L = ceil(Sk/n) rounded
        up to a multiple of 128 (reading: splits are whole kernel tiles)."""
        per = -(-sk // n)
        per = -(-per // 128) * 128
        return [(min(s * per, sk), min((s + 1) * per, sk)) for s in range(n)]

    def split_partials(self, n: int, rows=None):
        """Per split: o_s = (sum_j e^{s_ij - m_s} v_j) / l_s and
        lse_s = m_s + ln l_s over that split's keys (lse_s = -inf, o_s = 0 if no
        key)."""
        rows = np.arange(self.sq) if rows is None else np.asarray(rows)
        outs, lses = [], []
        for (k0, k1) in self.split_bounds(self.sk, n):
            cols = np.arange(k0, k1)
            if cols.size == 0:
                outs.append(np.zeros((rows.shape[0], self.dv)))
                lses.append(np.full(rows.shape[0], -np.inf))
                continue
            _, s = self.scores(rows, cols)
            p, lse = _probs(s, self.mask(rows, cols))
            outs.append(p @ self.v[cols])
            lses.append(lse)
        return np.stack(outs), np.stack(lses)


def combine_splits(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge split partials: LSE = ln sum_s e^{lse_s}; O = sum_s e^{lse_s - LSE} o_s.

    This is [PCB]'s pairwise merge (m_new = max, rescale by exp(m - m_new))
    applied to normalised partials. Empty splits (lse_s = -inf) weigh 0; all
    splits empty -> O = 0, LSE = -inf.
    """
    mx = np.max(lse_parts, axis=0)
    live = np.isfinite(mx)
    mx_safe = np.where(live, mx, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - mx_safe[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(live, mx_safe + np.log(np.where(live, tot, 1.0)), -np.inf)
    o = np.where(live[:, None],
                 np.einsum("sr,srd->rd", w, o_parts) / np.where(live, tot, 1.0)[:, None], 0.0)
    return o, lse


def _head_problem(q, k, v, b, h, spec):
    kb = spec.get("key_bias")
    return Problem(q[b, h], k[b, h], v[b, h], kind=spec.get("kind", NONE),
                   scale=spec.get("scale"), window_left=spec.get("window_left", -1),
                   block_size=spec.get("block_size", 0),
                   prefix_len=spec.get("prefix_len", 0), topk=spec.get("topk", 0),
                   rel_bias_slope=spec.get("rel_bias_slope", 0.0),
                   softcap=spec.get("softcap", 0.0), table=_head_table(spec, b, h),
                   key_bias=None if kb is None else kb[b, h])


def forward(q, k, v, spec: dict, heads=None, rows=None):
    """[B,H,S,D] forward over the listed (b, h) heads (default: all)."""
    B, H = q.shape[:2]
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    out = {}
    for (b, h) in heads:
        out[(b, h)] = _head_problem(q, k, v, b, h, spec).forward(rows)
    return out


def backward(q, k, v, do, spec: dict, heads=None, rows=None, cols=None):
    B, H = q.shape[:2]
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    out = {}
    for (b, h) in heads:
        out[(b, h)] = _head_problem(q, k, v, b, h, spec).backward(do[b, h], rows, cols)
    return out


def _head_table(spec: dict, b: int, h: int):
    """The element table of head (b, h): spec["table"] is [Sq, Sk] (shared)
    or [B, H, Sq, Sk]."""
    t = spec.get("table")
    if t is None:
        return None
    t = np.asarray(t, dtype=bool)
    return t if t.ndim == 2 else t[b, h]


def block_lists(B, H, sq, sk, spec: dict, sparse_m: int, sparse_n: int):
    """Block-sparse lists by brute-force enumeration of the element mask.

    [FA2C] builds, from one mask predicate, forward lists per q-block of
    k-blocks and backward lists per k-block of q-blocks, separating blocks
    that need the element mask ("partial") from blocks every pair of which is
    allowed ("full"); blocks with no allowed pair are absent. Reading: a block
    cut by the sequence end is never full; lists ascend; unused tail entries
    are 0; counts and indices are int32.
    """
    nqb = -(-sq // sparse_m)
    nkb = -(-sk // sparse_n)
    shape_f = (B, H, nqb)
    res = {
        "q_mask_cnt": np.zeros(shape_f, np.int32), "q_mask_idx": np.zeros(shape_f + (nkb,), np.int32),
        "q_full_cnt": np.zeros(shape_f, np.int32), "q_full_idx": np.zeros(shape_f + (nkb,), np.int32),
        "k_mask_cnt": np.zeros((B, H, nkb), np.int32), "k_mask_idx": np.zeros((B, H, nkb, nqb), np.int32),
        "k_full_cnt": np.zeros((B, H, nkb), np.int32), "k_full_idx": np.zeros((B, H, nkb, nqb), np.int32),
    }
    kb = spec.get("key_bias")
    rows = np.arange(sq)
    cols = np.arange(sk)
    for b in range(B):
        for h in range(H):
            keep = None
            if spec.get("kind", NONE) == DYNAMIC_TOPK:
                keep = topk_keep(np.asarray(kb[b, h], dtype=np.float64), spec.get("topk", 0))
            m = allowed(spec.get("kind", NONE), sq, sk, rows, cols,
                        window_left=spec.get("window_left", -1),
                        block_size=spec.get("block_size", 0),
                        prefix_len=spec.get("prefix_len", 0), keep=keep, table=_head_table(spec, b, h))
            pad = np.zeros((nqb * sparse_m, nkb * sparse_n), dtype=bool)
            pad[:sq, :sk] = m
            cnt = pad.reshape(nqb, sparse_m, nkb, sparse_n).sum(axis=(1, 3), dtype=np.int64)
            whole = np.zeros((nqb, nkb), dtype=bool)
            whole[: sq // sparse_m, : sk // sparse_n] = True
            full = whole & (cnt == sparse_m * sparse_n)
            part = (cnt > 0) & ~full
            for r in range(nqb):
                pl = np.nonzero(part[r])[0]
                fl = np.nonzero(full[r])[0]
                res["q_mask_cnt"][b, h, r] = pl.size
                res["q_mask_idx"][b, h, r, : pl.size] = pl
                res["q_full_cnt"][b, h, r] = fl.size
                res["q_full_idx"][b, h, r, : fl.size] = fl
            for c in range(nkb):
                pl = np.nonzero(part[:, c])[0]
                fl = np.nonzero(full[:, c])[0]
                res["k_mask_cnt"][b, h, c] = pl.size
                res["k_mask_idx"][b, h, c, : pl.size] = pl
                res["k_full_cnt"][b, h, c] = fl.size
                res["k_full_idx"][b, h, c, : fl.size] = fl
    return res


def keep_bits(key_bias, topk: int):
    """Dynamic keep set packed as uint32 words [B, H, ceil(Sk/32)], bit j%32 of
    word j//32 = key j kept."""
    B, H, sk = key_bias.shape
    nw = -(-sk // 32)
    out = np.zeros((B, H, nw), dtype=np.uint32)
    for b in range(B):
        for h in range(H):
            keep = topk_keep(np.asarray(key_bias[b, h], dtype=np.float64), topk)
            for j in np.nonzero(keep)[0]:
                out[b, h, j // 32] |= np.uint32(1) << np.uint32(j % 32)
    return out


def keep_index(key_bias, topk: int):
    """Kept-key index list [B, H, Sk] int32: per (b, h) the indices of the
    kept keys in ascending order, then 0 up to Sk (the library's gathered
    dynamic path streams exactly these keys)."""
    B, H, sk = key_bias.shape
    out = np.zeros((B, H, sk), dtype=np.int32)
    for b in range(B):
        for h in range(H):
            kept = np.nonzero(topk_keep(np.asarray(key_bias[b, h], dtype=np.float64), topk))[0]
            out[b, h, : kept.size] = kept
    return out


def pair_count(sq, sk, spec: dict, key_bias=None) -> int:
    """N = number of allowed (i, j) pairs of one head (the unmasked-FLOP count
    is 2 N (Dqk + Dv) forward and 2 N (3 Dqk + 2 Dv) backward)."""
    keep = None
    if spec.get("kind", NONE) == DYNAMIC_TOPK:
        keep = topk_keep(np.asarray(key_bias, dtype=np.float64), spec.get("topk", 0))
    total = 0
    cols = np.arange(sk)
    for r0 in range(0, sq, 1024):
        rows = np.arange(r0, min(sq, r0 + 1024))
        total += int(allowed(spec.get("kind", NONE), sq, sk, rows, cols,
                             window_left=spec.get("window_left", -1),
                             block_size=spec.get("block_size", 0),
                             prefix_len=spec.get("prefix_len", 0), keep=keep,
                             table=_head_table(spec, 0, 0)).sum())
    return total
