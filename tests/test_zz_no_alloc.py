"""attn_fwd_splitkv_noalloc: the split-KV decode entry point for callers that
cannot allocate device memory (for example a plug-in whose device memory all
belongs to a host engine's allocator, or a decode loop that must never call
cudaMalloc once it runs). Its split partials live in the library's own static
scratch array instead of a caller workspace.

The GPU tests call it through the C ABI twice in a row per case, with
different inputs and split counts, and check each result against
attn_fwd_splitkv given its own workspace (the same kernels: bit for bit) and
against the fp64 oracle within the bf16 tolerance the parity tests use. The
cases cover the per-row CUDA-core decode (Hkv = H), the packed tensor-core
decode of grouped query heads (Hkv < H, whose split partials then also live
in the static scratch) and a causal decode with several query rows. The file
is named to be collected last, and it works in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_tma_gb300 import binding as bd
from block_sparse_attention_tma_gb300.synth import make_inputs
from helpers import check_lse, check_out
from oracle import attention as orc

SCRATCH = 16 << 20  # GBATTN_NOALLOC_SCRATCH_BYTES


def _mask(causal):
    return bd.MaskSpec(kind=bd.CAUSAL if causal else bd.NONE).c()


def _call_noalloc(q, k, v, n, o, lse, causal):
    lib = bd.load_library()
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    m = _mask(causal)
    return lib.attn_fwd_splitkv_noalloc(bd.BF16, B, H, k.shape[1], Sq, Sk, D, D, q.data_ptr(), k.data_ptr(),
                                        v.data_ptr(), 0.0,
                                        ctypes.byref(m), n, o.data_ptr(), lse.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)


def _call_with_workspace(q, k, v, n, causal):
    lib = bd.load_library()
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = torch.empty(B, H, Sq, D, dtype=q.dtype, device=q.device)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    need = lib.attn_fwd_splitkv_workspace_bytes(B, H, Sq, D, n)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    m = _mask(causal)
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


# (B, H, Hkv, Sq, Sk, D, splits, causal): two calls in a row per case
CASES = {
    "per_row": ((4, 8, 8, 1, 4000, 128, 8, False), (2, 16, 16, 3, 2500, 64, 16, False)),
    "gqa_packed": ((2, 32, 8, 1, 3000, 128, 4, False), (3, 16, 4, 2, 1500, 64, 8, False)),
    "causal": ((2, 4, 4, 5, 700, 128, 4, True), (1, 8, 2, 3, 900, 64, 2, True)),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(name):
    dev = torch.device("cuda")
    for call, (B, H, Hkv, Sq, Sk, D, n, causal) in enumerate(CASES[name]):
        x = make_inputs(B, H, Sq, Sk, D, D, "bf16", seed=42 + call, dout=False, Hkv=Hkv)
        q, k, v = (x[t].to(dev) for t in ("q", "k", "v"))
        o = torch.full((B, H, Sq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device=dev)
        assert _call_noalloc(q, k, v, n, o, lse, causal) == 0
        o_ref, lse_ref = _call_with_workspace(q, k, v, n, causal)
        torch.cuda.synchronize()
        assert bd.load_library().gbattn_last_device_error(None) == 0
        assert not torch.isnan(o).any() and not torch.isnan(lse).any()
        # the fp64 oracle, head by head (query head h reads key/value head
        # h // (H / Hkv)), for both entry points
        f64 = lambda t: t.float().double().numpy()  # noqa: E731
        qh, kh, vh = f64(x["q"]), f64(x["k"]), f64(x["v"])
        G = H // Hkv
        for which, (oo, ll) in (("noalloc", (o, lse)), ("workspace", (o_ref, lse_ref))):
            og, lg = f64(oo.cpu()), ll.cpu().double().numpy()
            for b in range(B):
                for h in range(H):
                    p = orc.Problem(qh[b, h], kh[b, h // G], vh[b, h // G], kind=orc.CAUSAL if causal else orc.NONE)
                    o_r, l_r = p.forward()
                    check_out(og[b, h], o_r)
                    check_lse(lg[b, h], l_r)
        # same kernels, partials in another buffer: identical results
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
