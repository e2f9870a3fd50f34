"""attn_fwd_splitkv_noalloc: the split-KV decode entry point for callers that
cannot allocate device memory (for example a plug-in whose device memory all
belongs to a host engine's allocator, or a decode loop that must never call
cudaMalloc once it runs). Its split partials live in the library's own static
scratch array instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, with different inputs
and split counts, and checks each result against attn_fwd_splitkv given its
own workspace, within the bf16 tolerance the parity tests use. The file is
named to be collected last, and it works in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_tma_gb300 import binding as bd

SCRATCH = 16 << 20  # GBATTN_NOALLOC_SCRATCH_BYTES


def _call_noalloc(q, k, v, n, o, lse):
    lib = bd.load_library()
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    m = bd.MaskSpec().c()
    return lib.attn_fwd_splitkv_noalloc(bd.BF16, B, H, k.shape[1], Sq, Sk, D, D, q.data_ptr(), k.data_ptr(),
                                        v.data_ptr(), 0.0,
                                        ctypes.byref(m), n, o.data_ptr(), lse.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)


def _call_with_workspace(q, k, v, n):
    lib = bd.load_library()
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = torch.empty(B, H, Sq, D, dtype=q.dtype, device=q.device)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    need = lib.attn_fwd_splitkv_workspace_bytes(B, H, Sq, D, n)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    m = bd.MaskSpec().c()
    rc = lib.attn_fwd_splitkv(bd.BF16, B, H, k.shape[1], Sq, Sk, D, D, q.data_ptr(), k.data_ptr(), v.data_ptr(), 0.0,
                              ctypes.byref(m), n, o.data_ptr(), lse.data_ptr(), ws.data_ptr(), need,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    return o, lse


def test_rejects_problems_larger_than_the_scratch():
    lib = bd.load_library()
    fake = 1 << 20
    # 64 splits x 64 x 64 rows x 128 fp32 partials = 128 MiB > 16 MiB
    rc = lib.attn_fwd_splitkv_noalloc(bd.BF16, 64, 64, 64, 1, 65536, 128, 128, fake, fake, fake, 0.0, None, 64,
                                      fake, fake, None)
    assert rc == bd.ERR_WORKSPACE
    assert lib.attn_fwd_splitkv_workspace_bytes(64, 64, 1, 128, 64) > SCRATCH


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(42)
    for B, H, Sq, Sk, D, n in ((4, 8, 1, 4000, 128, 8), (2, 16, 3, 2500, 64, 16)):
        q = torch.randn(B, H, Sq, D, generator=g, device=dev).bfloat16()
        k = torch.randn(B, H, Sk, D, generator=g, device=dev).bfloat16()
        v = torch.randn(B, H, Sk, D, generator=g, device=dev).bfloat16()
        o = torch.full((B, H, Sq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device=dev)
        assert _call_noalloc(q, k, v, n, o, lse) == 0
        o_ref, lse_ref = _call_with_workspace(q, k, v, n)
        torch.cuda.synchronize()
        assert bd.load_library().gbattn_last_device_error(None) == 0
        a, r = o.double().cpu().numpy(), o_ref.double().cpu().numpy()
        assert not np.isnan(a).any()
        assert np.all(np.abs(a - r) <= 2e-2 + 2e-2 * np.abs(r))
        assert np.max(np.abs(lse.double().cpu().numpy() - lse_ref.double().cpu().numpy())) <= 2e-2
