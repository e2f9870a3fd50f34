"""The abort path of the kernels' bounded waits, on a real GPU, without a
fault or a hang: the test hook gbattn_test_fwd_stalled launches the bf16
forward kernel with a 1 ms wait limit and the first K tile of every CTA
withheld, so the MMA thread's wait for it runs out. The call must come back
in milliseconds, gbattn_last_device_error must report GBATTN_ERR_TIMEOUT once
(and clear it), and the next normal forward on the same GPU must match the
oracle (the kernel drained its copies and freed its tensor memory)."""
import ctypes
import time

import numpy as np
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga
from block_sparse_attention_tma_gb300 import binding as bd
from block_sparse_attention_tma_gb300.synth import make_inputs
from helpers import check_lse, check_out, f64
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
