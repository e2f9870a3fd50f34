"""Thin ctypes binding of libgbattn.so (argument marshalling only).

Every entry point has the name of its C counterpart in include/gbattn.h and
passes device pointers, sizes and the current CUDA stream straight through;
PyTorch only allocates the output / workspace tensors. There is no fallback:
if the library cannot be loaded, or a call returns an error status, a
GbattnError is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbattn.so")

NONE, CAUSAL, SLIDING, BLOCK_DIAG, PREFIX_LM, DYNAMIC_TOPK, MINI_CAUSAL, TABLE = range(8)
BF16, FP32 = 0, 1
_DT = {torch.bfloat16: BF16, torch.float32: FP32}

OK = 0
ERR_ARG, ERR_ALIGN, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_BLOCKS, ERR_CUDA, ERR_TIMEOUT = -1, -2, -3, -4, -5, -6, -7


class GbattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {code} ({strerror(code)})")


class _Mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("window_left", ctypes.c_int), ("block_size", ctypes.c_int),
                ("prefix_len", ctypes.c_int), ("topk", ctypes.c_int), ("rel_bias_slope", ctypes.c_float),
                ("softcap", ctypes.c_float), ("key_bias", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("table_per_head", ctypes.c_int)]


class _Blocks(ctypes.Structure):
    _fields_ = [("sparse_m", ctypes.c_int), ("sparse_n", ctypes.c_int)] + [
        (n, ctypes.c_void_p) for n in ("q_mask_cnt", "q_mask_idx", "q_full_cnt", "q_full_idx",
                                       "k_mask_cnt", "k_mask_idx", "k_full_cnt", "k_full_idx", "keep_bits",
                                       "keep_idx")]


_lib = None

# (name, restype, argtypes)
_SIGS = [
    ("gbattn_version", ctypes.c_int, []),
    ("gbattn_strerror", ctypes.c_char_p, [ctypes.c_int]),
    ("gbattn_block_mask_sizes", ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_size_t)] * 6),
    ("build_block_mask", ctypes.c_int, [ctypes.c_int] * 4 + [ctypes.POINTER(_Mask), ctypes.POINTER(_Blocks),
                                                              ctypes.c_void_p]),
    ("attn_fwd", ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.c_void_p] * 3 + [ctypes.c_float, ctypes.POINTER(_Mask),
                                                                              ctypes.POINTER(_Blocks),
                                                                              ctypes.c_void_p, ctypes.c_void_p,
                                                                              ctypes.c_void_p]),
    ("attn_bwd_workspace_bytes", ctypes.c_size_t, [ctypes.c_int] * 7),
    ("attn_bwd", ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.c_void_p] * 6 + [ctypes.c_float, ctypes.POINTER(_Mask),
                                                                              ctypes.POINTER(_Blocks), ctypes.c_int]
     + [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p]),
    ("attn_fwd_splitkv_workspace_bytes", ctypes.c_size_t, [ctypes.c_int] * 5),
    ("attn_fwd_splitkv", ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.c_void_p] * 3 + [ctypes.c_float,
                                                                                      ctypes.POINTER(_Mask),
                                                                                      ctypes.c_int]
     + [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]),
    ("attn_fwd_splitkv_paged", ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.c_void_p] * 3
     + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float,
        ctypes.POINTER(_Mask), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_void_p]),
    ("attn_fwd_splitkv_noalloc", ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.c_void_p] * 3
     + [ctypes.c_float, ctypes.POINTER(_Mask), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("gbattn_last_device_error", ctypes.c_int, [ctypes.c_void_p]),
    ("gbattn_set_dkdv_cta_pair", ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    # include/gbattn_test.h: a test hook, not part of the attention API
    ("gbattn_test_fwd_stalled", ctypes.c_int, [ctypes.c_int] * 5 + [ctypes.c_void_p] * 5
     + [ctypes.c_ulonglong, ctypes.c_void_p]),
    ("gbattn_test_bwd_stalled", ctypes.c_int, [ctypes.c_int] * 4 + [ctypes.c_void_p] * 10
     + [ctypes.c_size_t, ctypes.c_ulonglong, ctypes.c_void_p]),
]

EXPORTS = [s[0] for s in _SIGS]


def load_library(path: str = LIB_PATH):
    """Loads libgbattn.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise GbattnError(ERR_CUDA, f"libgbattn.so not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, res, args in _SIGS:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load_library().gbattn_strerror(code).decode()
    except Exception:  # the library itself may be what is missing
        return "unknown"


def _check(rc: int, what: str):
    if rc != OK:
        raise GbattnError(rc, what)


def _check_tensors(what: str, specs, device_of: Optional[torch.Tensor] = None):
    """Checks the tensors of one call before any pointer crosses the C ABI,
    which takes raw pointers and derives sizes from the shapes given to it.

    specs: (name, tensor or None, expected shape (None = any, an int entry of
    None = any size there), allowed dtypes). Every given tensor must be
    contiguous, have the expected shape and dtype, and sit on the same CUDA
    device as `device_of` (default: the first given tensor). Raises ValueError.
    """
    ref = device_of
    for name, t, shape, dtypes in specs:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{what}: {name} must be a torch.Tensor")
        if shape is not None:
            ok = t.dim() == len(shape) and all(e is None or e == d for e, d in zip(shape, t.shape))
            if not ok:
                want = "[" + ", ".join("*" if e is None else str(e) for e in shape) + "]"
                raise ValueError(f"{what}: {name} has shape {list(t.shape)}, expected {want}")
        if dtypes is not None and t.dtype not in dtypes:
            raise ValueError(f"{what}: {name} has dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")
        if not t.is_contiguous():
            raise ValueError(f"{what}: {name} must be contiguous")
        if ref is None:
            ref = t
    for name, t, _, _ in specs:
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"{what}: {name} must be on a CUDA device (is on {t.device})")
        if t.device != ref.device:
            raise ValueError(f"{what}: {name} is on {t.device}, the other tensors on {ref.device}")


_FLOAT = (torch.bfloat16, torch.float32)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


def _qkv_dims(what, q, k, v):
    """Reads B, H, Hkv, Sq, Sk, Dqk, Dv off the q / k / v trio and returns
    them with the trio's check specs (for one _check_tensors call, so that
    every shape is checked before any device)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError(f"{what}: {name} must be a 4-D tensor [B, heads, S, D]")
    B, H, Sq, Dqk = q.shape
    Hkv, Sk, Dv = k.shape[1], k.shape[2], v.shape[3]
    if q.dtype not in _FLOAT:
        raise ValueError(f"{what}: q has dtype {q.dtype}, expected bfloat16 or float32")
    specs = [("q", q, None, None), ("k", k, (B, Hkv, Sk, Dqk), (q.dtype,)), ("v", v, (B, Hkv, Sk, Dv), (q.dtype,))]
    return (B, H, Hkv, Sq, Sk, Dqk, Dv), specs


def _mask_tensors(what, mask, B, H, Sq, Sk):
    if mask is None:
        return []
    nw = (Sk + 31) // 32
    out = [("mask.key_bias", mask.key_bias, (B, H, Sk), _F32)]
    if mask.table is not None:
        shape = (Sq, nw) if mask.table.dim() == 2 else (B, H, Sq, nw)
        out.append(("mask.table", mask.table, shape, _I32))
    return out


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


@dataclass
class MaskSpec:
    kind: int = NONE
    window_left: int = -1
    block_size: int = 0
    prefix_len: int = 0
    topk: int = 0
    rel_bias_slope: float = 0.0
    softcap: float = 0.0
    key_bias: Optional[torch.Tensor] = None  # [B, H, Sk] fp32 on the GPU
    table: Optional[torch.Tensor] = None     # TABLE: int32 bits [Sq, ceil(Sk/32)] or [B, H, Sq, ceil(Sk/32)]

    def c(self) -> _Mask:
        return _Mask(self.kind, self.window_left, self.block_size, self.prefix_len, self.topk,
                     float(self.rel_bias_slope), float(self.softcap),
                     None if self.key_bias is None else self.key_bias.data_ptr(),
                     None if self.table is None else self.table.data_ptr(),
                     0 if self.table is None or self.table.dim() == 2 else 1)


def pack_mask_table(allowed: torch.Tensor) -> torch.Tensor:
    """Packs a boolean element mask [..., Sq, Sk] into the TABLE kind's bits:
    int32 words [..., Sq, ceil(Sk/32)], bit j % 32 of word j // 32 = pair
    (i, j) allowed. Runs on the tensor's device (torch ops, no attention
    arithmetic)."""
    *lead, sq, sk = allowed.shape
    nw = (sk + 31) // 32
    pad = torch.zeros(*lead, sq, nw * 32, dtype=torch.int64, device=allowed.device)
    pad[..., :sk] = allowed.to(torch.int64)
    w = pad.view(*lead, sq, nw, 32) << torch.arange(32, device=allowed.device, dtype=torch.int64)
    packed = w.sum(-1)  # < 2^32
    return (packed - (packed >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32).contiguous()


@dataclass
class BlockLists:
    sparse_m: int
    sparse_n: int
    tensors: dict = field(default_factory=dict)  # name -> int32 / uint32-as-int32 tensor

    def c(self) -> _Blocks:
        b = _Blocks(self.sparse_m, self.sparse_n)
        for name, t in self.tensors.items():
            setattr(b, name, t.data_ptr())
        return b


def _list_tensors(lists: Optional[BlockLists]):
    if lists is None:
        return []
    return [(f"lists.{n}", t, None, _I32) for n, t in lists.tensors.items()]


def alloc_block_lists(B, H, Sq, Sk, sparse_m, sparse_n, device="cuda", gather=True) -> BlockLists:
    """Allocates every list array. gather=True also allocates the dynamic
    mask's kept-key index list, with which the bf16 kernels stream only the
    kept keys; gather=False leaves it NULL (the kernels then walk the lists
    and test the keep bits)."""
    lib = load_library()
    sz = [ctypes.c_size_t() for _ in range(6)]
    _check(lib.gbattn_block_mask_sizes(B, H, Sq, Sk, sparse_m, sparse_n, *[ctypes.byref(s) for s in sz]),
           "gbattn_block_mask_sizes")
    qc, qi, kc, ki, kw, kx = (s.value // 4 for s in sz)
    mk = lambda n: torch.empty(max(n, 1), dtype=torch.int32, device=device)  # noqa: E731
    t = {"q_mask_cnt": mk(qc), "q_mask_idx": mk(qi), "q_full_cnt": mk(qc), "q_full_idx": mk(qi),
         "k_mask_cnt": mk(kc), "k_mask_idx": mk(ki), "k_full_cnt": mk(kc), "k_full_idx": mk(ki),
         "keep_bits": mk(kw)}
    if gather:
        t["keep_idx"] = mk(kx)
    return BlockLists(sparse_m, sparse_n, t)


def build_block_mask(B, H, Sq, Sk, mask: MaskSpec, lists: BlockLists, stream=None) -> BlockLists:
    lib = load_library()
    _check_tensors("build_block_mask", _mask_tensors("build_block_mask", mask, B, H, Sq, Sk) + _list_tensors(lists))
    cm, cb = mask.c(), lists.c()
    _check(lib.build_block_mask(B, H, Sq, Sk, ctypes.byref(cm), ctypes.byref(cb), _stream(stream)),
           "build_block_mask")
    return lists


def attn_fwd(q, k, v, scale=0.0, mask: Optional[MaskSpec] = None, lists: Optional[BlockLists] = None,
             o=None, lse=None, stream=None):
    """q [B, H, Sq, Dqk]; k, v [B, Hkv, Sk, D] (Hkv divides H: grouped-query
    attention when Hkv < H)."""
    lib = load_library()
    (B, H, Hkv, Sq, Sk, Dqk, Dv), qkv = _qkv_dims("attn_fwd", q, k, v)
    _check_tensors("attn_fwd", qkv + [("o", o, (B, H, Sq, Dv), (q.dtype,)), ("lse", lse, (B, H, Sq), _F32)]
                   + _mask_tensors("attn_fwd", mask, B, H, Sq, Sk) + _list_tensors(lists), device_of=q)
    if o is None:
        o = torch.empty(B, H, Sq, Dv, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    mask = mask or MaskSpec()
    cm = mask.c()
    cb = lists.c() if lists is not None else None
    _check(lib.attn_fwd(_DT.get(q.dtype, -1), B, H, Hkv, Sq, Sk, Dqk, Dv, _ptr(q), _ptr(k), _ptr(v), float(scale),
                        ctypes.byref(cm), ctypes.byref(cb) if cb is not None else None, _ptr(o), _ptr(lse),
                        _stream(stream)), "attn_fwd")
    return o, lse


def attn_bwd_workspace_bytes(dtype, B, H, Sq, Sk, Dqk, Dv) -> int:
    return int(load_library().attn_bwd_workspace_bytes(_DT.get(dtype, -1), B, H, Sq, Sk, Dqk, Dv))


def attn_bwd(q, k, v, o, dout, lse, scale=0.0, mask: Optional[MaskSpec] = None,
             lists: Optional[BlockLists] = None, deterministic=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None, dkey_bias: Optional[torch.Tensor] = None):
    """Returns (dq, dk, dv); when dkey_bias (fp32 [B, H, Sk] on the GPU) is
    given it receives the gradient of the key bias."""
    lib = load_library()
    (B, H, Hkv, Sq, Sk, Dqk, Dv), qkv = _qkv_dims("attn_bwd", q, k, v)
    _check_tensors("attn_bwd", qkv + [("o", o, (B, H, Sq, Dv), (q.dtype,)), ("dout", dout, (B, H, Sq, Dv), (q.dtype,)),
                                ("lse", lse, (B, H, Sq), _F32), ("dq", dq, (B, H, Sq, Dqk), (q.dtype,)),
                                ("dk", dk, (B, Hkv, Sk, Dqk), (q.dtype,)), ("dv", dv, (B, Hkv, Sk, Dv), (q.dtype,)),
                                ("dkey_bias", dkey_bias, (B, H, Sk), _F32), ("workspace", workspace, None, None)]
                   + _mask_tensors("attn_bwd", mask, B, H, Sq, Sk) + _list_tensors(lists), device_of=q)
    if o is None or dout is None or lse is None:
        raise ValueError("attn_bwd: o, dout and lse are required")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_bwd_workspace_bytes(q.dtype, B, H, Sq, Sk, Dqk, Dv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    mask = mask or MaskSpec()
    cm = mask.c()
    cb = lists.c() if lists is not None else None
    _check(lib.attn_bwd(_DT.get(q.dtype, -1), B, H, Hkv, Sq, Sk, Dqk, Dv, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                        _ptr(dout),
                        _ptr(lse), float(scale), ctypes.byref(cm), ctypes.byref(cb) if cb is not None else None,
                        int(bool(deterministic)), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dkey_bias), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream)), "attn_bwd")
    return dq, dk, dv


def attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits) -> int:
    return int(load_library().attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits))


def attn_fwd_splitkv(q, k, v, scale=0.0, mask: Optional[MaskSpec] = None, num_splits=1, o=None, lse=None,
                     workspace=None, stream=None):
    lib = load_library()
    (B, H, Hkv, Sq, Sk, Dqk, Dv), qkv = _qkv_dims("attn_fwd_splitkv", q, k, v)
    _check_tensors("attn_fwd_splitkv", qkv + [("o", o, (B, H, Sq, Dv), (q.dtype,)), ("lse", lse, (B, H, Sq), _F32),
                                        ("workspace", workspace, None, None)], device_of=q)
    if o is None:
        o = torch.empty(B, H, Sq, Dv, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    need = attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    mask = mask or MaskSpec()
    cm = mask.c()
    _check(lib.attn_fwd_splitkv(_DT.get(q.dtype, -1), B, H, Hkv, Sq, Sk, Dqk, Dv, _ptr(q), _ptr(k), _ptr(v),
                                float(scale), ctypes.byref(cm), int(num_splits), _ptr(o), _ptr(lse), _ptr(workspace),
                                0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _stream(stream)), "attn_fwd_splitkv")
    return o, lse


def attn_fwd_splitkv_paged(q, k_cache, v_cache, page_table, seqlens_k, scale=0.0, mask: Optional[MaskSpec] = None,
                           num_splits=1, o=None, lse=None, workspace=None, stream=None):
    """Split-KV decode over a paged cache: k_cache / v_cache [num_pages, Hkv,
    page_size, D] bf16, page_table [B, max_pages] int32 and seqlens_k [B]
    int32 on the GPU."""
    lib = load_library()
    what = "attn_fwd_splitkv_paged"
    for name, t, nd in (("q", q, 4), ("k_cache", k_cache, 4), ("v_cache", v_cache, 4), ("page_table", page_table, 2),
                        ("seqlens_k", seqlens_k, 1)):
        if not isinstance(t, torch.Tensor) or t.dim() != nd:
            raise ValueError(f"{what}: {name} must be a {nd}-D tensor")
    B, H, Sq, Dqk = q.shape
    num_pages, Hkv, page_size, Dv = v_cache.shape
    max_pages = page_table.shape[1]
    _check_tensors(what, [("q", q, None, _FLOAT), ("k_cache", k_cache, (num_pages, Hkv, page_size, Dqk), (q.dtype,)),
                          ("v_cache", v_cache, None, (q.dtype,)), ("page_table", page_table, (B, max_pages), _I32),
                          ("seqlens_k", seqlens_k, (B,), _I32), ("o", o, (B, H, Sq, Dv), (q.dtype,)),
                          ("lse", lse, (B, H, Sq), _F32), ("workspace", workspace, None, None)], device_of=q)
    if o is None:
        o = torch.empty(B, H, Sq, Dv, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    need = attn_fwd_splitkv_workspace_bytes(B, H, Sq, Dv, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    mask = mask or MaskSpec()
    cm = mask.c()
    _check(lib.attn_fwd_splitkv_paged(_DT.get(q.dtype, -1), B, H, Hkv, Sq, Dqk, Dv, _ptr(q), _ptr(k_cache),
                                      _ptr(v_cache), num_pages, page_size, _ptr(page_table), max_pages,
                                      _ptr(seqlens_k), float(scale), ctypes.byref(cm), int(num_splits), _ptr(o),
                                      _ptr(lse), _ptr(workspace),
                                      0 if workspace is None else workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "attn_fwd_splitkv_paged")
    return o, lse


def set_dkdv_cta_pair(mode: int) -> int:
    """Selects attn_bwd's dK/dV kernel where the CTA-pair kernel applies: 1 =
    CTA pair, 0 = one CTA, -1 = library default. Returns the previous mode."""
    prev = ctypes.c_int(0)
    _check(load_library().gbattn_set_dkdv_cta_pair(int(mode), ctypes.byref(prev)), "gbattn_set_dkdv_cta_pair")
    return prev.value


def last_device_error(stream=None) -> int:
    return int(load_library().gbattn_last_device_error(_stream(stream)))


def attn_fwd_splitkv_noalloc(q, k, v, scale=0.0, mask: Optional[MaskSpec] = None, num_splits=1, o=None, lse=None,
                             stream=None):
    """attn_fwd_splitkv without a workspace argument, for callers that may not
    allocate device memory: the split partials go to the library's own static
    scratch array (limit GBATTN_NOALLOC_SCRATCH_BYTES, 16 MiB). Calls whose GPU
    work overlaps race on that array. Pass preallocated o / lse to allocate
    nothing here either."""
    lib = load_library()
    (B, H, Hkv, Sq, Sk, Dqk, Dv), qkv = _qkv_dims("attn_fwd_splitkv_noalloc", q, k, v)
    _check_tensors("attn_fwd_splitkv_noalloc", qkv + [("o", o, (B, H, Sq, Dv), (q.dtype,)), ("lse", lse, (B, H, Sq), _F32)],
                   device_of=q)
    if o is None:
        o = torch.empty(B, H, Sq, Dv, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    mask = mask or MaskSpec()
    cm = mask.c()
    _check(lib.attn_fwd_splitkv_noalloc(_DT.get(q.dtype, -1), B, H, Hkv, Sq, Sk, Dqk, Dv, _ptr(q), _ptr(k), _ptr(v),
                                        float(scale), ctypes.byref(cm), int(num_splits), _ptr(o), _ptr(lse),
                                        _stream(stream)), "attn_fwd_splitkv_noalloc")
    return o, lse
