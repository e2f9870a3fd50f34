"""The C ABI without a GPU: the library loads, exports every function that
include/gbattn.h declares, and rejects bad arguments on the host (before any
CUDA call) with the documented status codes."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT
import block_sparse_attention_tma_gb300 as ga
from block_sparse_attention_tma_gb300 import binding as bd

HEADER = os.path.join(ROOT, "include", "gbattn.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def declared_functions():
    """Every function declared in include/*.h (the API header and the test
    hooks' header)."""
    src = "\n".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_fwd_splitkv", "build_block_mask", "gbattn_strerror",
              "gbattn_last_device_error", "gbattn_block_mask_sizes", "attn_bwd_workspace_bytes",
              "attn_fwd_splitkv_workspace_bytes", "gbattn_version"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ga.load_library()
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(bd.EXPORTS) >= set(declared_functions())
    assert "gbattn_test_fwd_stalled" in declared_functions()
    assert "gbattn_test_bwd_stalled" in declared_functions()
    assert lib.gbattn_version() == 102


def test_strerror_covers_codes():
    lib = ga.load_library()
    for c in range(0, -8, -1):
        assert lib.gbattn_strerror(c) not in (None, b"unknown status")


def test_block_mask_sizes():
    lib = ga.load_library()
    sz = [ctypes.c_size_t() for _ in range(6)]
    rc = lib.gbattn_block_mask_sizes(1, 16, 16384, 16384, 256, 512, *[ctypes.byref(s) for s in sz])
    assert rc == 0
    assert [s.value for s in sz] == [16 * 64 * 4, 16 * 64 * 32 * 4, 16 * 32 * 4, 16 * 32 * 64 * 4, 16 * 512 * 4,
                                     16 * 16384 * 4]
    assert lib.gbattn_block_mask_sizes(1, 1, 100, 100, 100, 128, *[None] * 6) == bd.ERR_ARG
    assert lib.gbattn_block_mask_sizes(0, 1, 100, 100, 128, 128, *[None] * 6) == bd.ERR_ARG


def test_workspace_queries():
    lib = ga.load_library()
    # 2 row vectors of [2,8,2048] fp32 (rows padded to 128)
    assert lib.attn_bwd_workspace_bytes(0, 2, 8, 2048, 2048, 64, 64) == 2 * 2 * 8 * 2048 * 4
    assert lib.attn_bwd_workspace_bytes(0, 1, 1, 100, 100, 64, 64) == 2 * 512
    assert lib.attn_bwd_workspace_bytes(0, 0, 8, 2048, 2048, 64, 64) == 0
    assert lib.attn_fwd_splitkv_workspace_bytes(32, 32, 1, 128, 1) == 0
    assert lib.attn_fwd_splitkv_workspace_bytes(32, 32, 1, 128, 4) == 4 * 1024 * 128 * 4 + 4 * 1024 * 4
    assert lib.attn_fwd_splitkv_workspace_bytes(32, 32, 1, 128, 65) == 0


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


def _fwd(dtype=0, B=1, H=1, Sq=128, Sk=128, Dqk=64, Dv=64, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE,
         mask=None, blocks=None, Hkv=None):
    lib = ga.load_library()
    m = mask.c() if mask is not None else None
    return lib.attn_fwd(dtype, B, H, H if Hkv is None else Hkv, Sq, Sk, Dqk, Dv, q, k, v, 0.0,
                        ctypes.byref(m) if m else None,
                        ctypes.byref(blocks) if blocks else None, o, lse, None)


def test_fwd_argument_checks():
    assert _fwd(B=0) == bd.ERR_ARG
    assert _fwd(H=4, Hkv=3) == bd.ERR_ARG   # Hkv must divide H
    assert _fwd(H=4, Hkv=0) == bd.ERR_ARG
    assert _fwd(H=4, Hkv=8) == bd.ERR_ARG
    assert _fwd(Sk=-1) == bd.ERR_ARG
    assert _fwd(q=0) == bd.ERR_ARG
    assert _fwd(q=FAKE + 8) == bd.ERR_ALIGN
    assert _fwd(Dqk=96, Dv=96) == bd.ERR_UNSUPPORTED      # bf16 head dims
    assert _fwd(Dqk=128, Dv=64) == bd.ERR_UNSUPPORTED
    assert _fwd(dtype=7) == bd.ERR_UNSUPPORTED
    assert _fwd(dtype=1, Dqk=200, Dv=8) == bd.ERR_UNSUPPORTED  # fp32 path: <= 128
    assert _fwd(mask=bd.MaskSpec(kind=9)) == bd.ERR_ARG
    assert _fwd(mask=bd.MaskSpec(kind=bd.BLOCK_DIAG, block_size=0)) == bd.ERR_ARG
    assert _fwd(mask=bd.MaskSpec(kind=bd.CAUSAL, softcap=-1.0)) == bd.ERR_ARG
    # a masked call needs block lists
    assert _fwd(mask=bd.MaskSpec(kind=bd.CAUSAL)) == bd.ERR_BLOCKS
    blk = bd._Blocks(256, 100)
    assert _fwd(mask=bd.MaskSpec(kind=bd.CAUSAL), blocks=blk) == bd.ERR_BLOCKS
    blk = bd._Blocks(256, 512)  # right tiles, but no list pointers
    assert _fwd(mask=bd.MaskSpec(kind=bd.CAUSAL), blocks=blk) == bd.ERR_BLOCKS


def test_valid_call_without_gpu_reports_unsupported_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd() == bd.ERR_UNSUPPORTED


def test_bwd_and_splitkv_argument_checks():
    lib = ga.load_library()
    args = [0, 1, 1, 1, 128, 128, 64, 64] + [FAKE] * 6 + [0.0, None, None]
    assert lib.attn_bwd(*args, 2, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == bd.ERR_ARG   # deterministic flag
    assert lib.attn_bwd(*args, 0, FAKE, FAKE, FAKE, None, None, 1 << 30, None) == bd.ERR_WORKSPACE
    assert lib.attn_bwd(*args, 0, FAKE, FAKE, FAKE, None, FAKE, 16, None) == bd.ERR_WORKSPACE
    assert lib.attn_bwd(*args, 0, FAKE, FAKE, FAKE, FAKE + 2, FAKE, 1 << 30, None) == bd.ERR_ALIGN  # dkey_bias
    gqa = [0, 1, 4, 2] + args[4:]
    assert lib.attn_bwd(*gqa, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == bd.ERR_UNSUPPORTED  # dkey_bias + GQA
    sk = [0, 32, 32, 32, 1, 65536, 128, 128, FAKE, FAKE, FAKE, 0.0, None]
    assert lib.attn_fwd_splitkv(*sk, 0, FAKE, FAKE, None, 0, None) == bd.ERR_ARG          # 0 splits
    assert lib.attn_fwd_splitkv(*sk, 4, FAKE, FAKE, None, 0, None) == bd.ERR_WORKSPACE
    m = bd.MaskSpec(kind=bd.SLIDING, window_left=3).c()
    sk2 = sk[:12] + [ctypes.byref(m)]
    assert lib.attn_fwd_splitkv(*sk2, 1, FAKE, FAKE, None, 0, None) == bd.ERR_UNSUPPORTED
    sk3 = list(sk)
    sk3[0] = 1
    assert lib.attn_fwd_splitkv(*sk3, 1, FAKE, FAKE, None, 0, None) == bd.ERR_UNSUPPORTED  # fp32 decode
    # paged decode: page size a multiple of 64, page table and key counts required
    pg = lambda **kw: lib.attn_fwd_splitkv_paged(  # noqa: E731
        0, 2, 8, kw.get("Hkv", 2), 1, 128, 128, FAKE, FAKE, FAKE, kw.get("num_pages", 16), kw.get("page_size", 256),
        kw.get("table", FAKE), 8, kw.get("seqlens", FAKE), 0.0, None, kw.get("splits", 1), FAKE, FAKE, None, 0, None)
    assert pg(page_size=100) == bd.ERR_ARG
    assert pg(page_size=32) == bd.ERR_ARG
    assert pg(table=None) == bd.ERR_ARG
    assert pg(seqlens=None) == bd.ERR_ARG
    assert pg(num_pages=0) == bd.ERR_ARG
    assert pg(Hkv=3) == bd.ERR_ARG
    assert pg(table=FAKE + 2) == bd.ERR_ALIGN
    assert pg(splits=4) == bd.ERR_WORKSPACE


def test_build_block_mask_argument_checks():
    lib = ga.load_library()
    m = bd.MaskSpec(kind=bd.DYNAMIC_TOPK, topk=4).c()  # no key bias
    b = bd._Blocks(128, 128, *[FAKE] * 9)
    assert lib.build_block_mask(1, 1, 128, 128, ctypes.byref(m), ctypes.byref(b), None) == bd.ERR_ARG
    m = bd.MaskSpec(kind=bd.CAUSAL).c()
    b = bd._Blocks(128, 128, *[FAKE] * 8, None)
    assert lib.build_block_mask(1, 1, 128, 128, ctypes.byref(m), None, None) == bd.ERR_ARG
    b2 = bd._Blocks(64, 128, *[FAKE] * 9)
    assert lib.build_block_mask(1, 1, 128, 128, ctypes.byref(m), ctypes.byref(b2), None) == bd.ERR_BLOCKS


def test_stalled_forward_hook_rejects_bad_arguments_on_the_host():
    lib = ga.load_library()
    f = FAKE
    assert lib.gbattn_test_fwd_stalled(1, 1, 128, 128, 64, f, f, f, f, f, 0, None) == bd.ERR_ARG  # wait 0
    assert lib.gbattn_test_fwd_stalled(1, 1, 128, 128, 64, f, f, f, f, f, 3 * 10**9, None) == bd.ERR_ARG
    assert lib.gbattn_test_fwd_stalled(1, 1, 128, 128, 64, f + 2, f, f, f, f, 10**6, None) == bd.ERR_ALIGN
    assert lib.gbattn_test_fwd_stalled(1, 1, 128, 128, 96, f, f, f, f, f, 10**6, None) == bd.ERR_UNSUPPORTED
    assert lib.gbattn_test_fwd_stalled(0, 1, 128, 128, 64, f, f, f, f, f, 10**6, None) == bd.ERR_ARG


def test_stalled_backward_hook_rejects_bad_arguments_on_the_host():
    lib = ga.load_library()
    f = FAKE
    ws = 1 << 30
    args = lambda B=1, D=64, q=f, wsb=ws, wait=10**6: (B, 1, 128, D, q, f, f, f, f, f, f, f, f, f, wsb, wait, None)
    assert lib.gbattn_test_bwd_stalled(*args(wait=0)) == bd.ERR_ARG
    assert lib.gbattn_test_bwd_stalled(*args(wait=3 * 10**9)) == bd.ERR_ARG
    assert lib.gbattn_test_bwd_stalled(*args(q=f + 2)) == bd.ERR_ALIGN
    assert lib.gbattn_test_bwd_stalled(*args(D=96)) == bd.ERR_UNSUPPORTED
    assert lib.gbattn_test_bwd_stalled(*args(B=0)) == bd.ERR_ARG
    assert lib.gbattn_test_bwd_stalled(*args(wsb=16)) == bd.ERR_WORKSPACE


def test_dkdv_cta_pair_selector_host_side():
    lib = ga.load_library()
    prev = ctypes.c_int(99)
    assert lib.gbattn_set_dkdv_cta_pair(1, ctypes.byref(prev)) == bd.OK
    first = prev.value
    assert first in (-1, 0, 1)
    assert lib.gbattn_set_dkdv_cta_pair(0, ctypes.byref(prev)) == bd.OK and prev.value == 1
    assert lib.gbattn_set_dkdv_cta_pair(2, ctypes.byref(prev)) == bd.ERR_ARG and prev.value == 1  # unchanged
    assert lib.gbattn_set_dkdv_cta_pair(-2, None) == bd.ERR_ARG
    assert lib.gbattn_set_dkdv_cta_pair(first, ctypes.byref(prev)) == bd.OK and prev.value == 0
    assert ga.set_dkdv_cta_pair(first) == first
