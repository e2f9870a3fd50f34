"""The abort path of the kernels' bounded waits, on a real GPU, without a
fault or a hang: the test hook gbattn_test_fwd_stalled launches the bf16
forward kernel with a 1 ms wait limit and the first K tile of every CTA
withheld, so the MMA thread's wait for it runs out; gbattn_test_bwd_stalled
does the same to the backward (the first dO tile of every dK/dV CTA and the
first K tile of every dQ CTA withheld: both MMA issuers of each kernel wait
for them). The call must come back in milliseconds, gbattn_last_device_error
must report GBATTN_ERR_TIMEOUT once (and clear it), and the next normal call
on the same GPU must match the oracle (the kernels drained their copies and
products and freed their tensor memory)."""
import ctypes
import time

import numpy as np
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga
from block_sparse_attention_tma_gb300 import binding as bd
from block_sparse_attention_tma_gb300.synth import make_inputs
from helpers import check_grad, check_lse, check_out, f64
from oracle import attention as orc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_stalled_forward_times_out_reports_and_recovers(D):
    lib = bd.load_library()
    B, H, S = 1, 4, 700
    x = make_inputs(B, H, S, S, D, D, "bf16", seed=42, dout=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.zeros(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, S, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.gbattn_last_device_error(None) == 0  # nothing pending from earlier tests
    t0 = time.time()
    rc = lib.gbattn_test_fwd_stalled(B, H, S, S, D, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), 1_000_000, ctypes.c_void_p(st))
    assert rc == bd.OK
    torch.cuda.synchronize()
    took = time.time() - t0
    assert took < 1.0, f"stalled launch took {took:.3f} s: the 1 ms limit did not apply"
    assert lib.gbattn_last_device_error(None) == bd.ERR_TIMEOUT
    assert lib.gbattn_last_device_error(None) == 0  # read and cleared
    # the context and the SMs are fine: a normal call right after is correct
    o2, lse2 = ga.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert lib.gbattn_last_device_error(None) == 0
    for h in range(H):
        o_ref, l_ref = orc.Problem(f64(x["q"][0, h]), f64(x["k"][0, h]), f64(x["v"][0, h])).forward()
        check_out(f64(o2[0, h]), o_ref)
        check_lse(f64(lse2[0, h]), l_ref)


@pytest.mark.parametrize("D", [64, 128])
def test_stalled_backward_times_out_reports_and_recovers(D):
    lib = bd.load_library()
    B, H, S = 1, 4, 700
    x = make_inputs(B, H, S, S, D, D, "bf16", seed=43)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = ga.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    nws = ga.attn_bwd_workspace_bytes(torch.bfloat16, B, H, S, S, D, D)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.gbattn_last_device_error(None) == 0
    t0 = time.time()
    rc = lib.gbattn_test_bwd_stalled(B, H, S, D, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                     ws.data_ptr(), nws, 1_000_000, ctypes.c_void_p(st))
    assert rc == bd.OK
    torch.cuda.synchronize()
    took = time.time() - t0
    assert took < 1.0, f"stalled backward took {took:.3f} s: the 1 ms limit did not apply"
    assert lib.gbattn_last_device_error(None) == bd.ERR_TIMEOUT
    assert lib.gbattn_last_device_error(None) == 0
    # a normal backward right after is correct
    dq2, dk2, dv2 = ga.attn_bwd(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    assert lib.gbattn_last_device_error(None) == 0
    for h in range(H):
        p = orc.Problem(f64(x["q"][0, h]), f64(x["k"][0, h]), f64(x["v"][0, h]))
        dq_r, dk_r, dv_r, _ = p.backward(f64(x["do"][0, h]))
        check_grad(f64(dq2[0, h]), dq_r, "dQ")
        check_grad(f64(dk2[0, h]), dk_r, "dK")
        check_grad(f64(dv2[0, h]), dv_r, "dV")
