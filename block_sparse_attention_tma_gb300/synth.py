"""Seeded synthetic inputs shared by the tests, the benchmark and smoke().

Holds no attention arithmetic: it only draws random tensors. A CPU
``torch.Generator`` seeded with 42 (the seed of the forward/backward runs in
"Optimize Flash Dynamic Mask Attention Kernel Configurations", Test
Configuration) draws, in this order, Q, K, V, dO and the key bias, each as
fp32 N(0, 1); Q/K/V/dO are then rounded to the run dtype, the bias stays fp32.
Both the CUDA path and the fp64 oracle read these very values (the oracle
widens them exactly).
"""
from __future__ import annotations

import torch

DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


def make_inputs(B, H, Sq, Sk, Dqk, Dv, dtype="bf16", seed=42, dout=True, bias=False, Hkv=None):
    """Hkv (default H): key/value heads, for grouped-query inputs."""
    g = torch.Generator().manual_seed(int(seed))
    td = DTYPES[dtype]
    Hkv = H if Hkv is None else Hkv
    out = {
        "q": torch.randn(B, H, Sq, Dqk, generator=g).to(td),
        "k": torch.randn(B, Hkv, Sk, Dqk, generator=g).to(td),
        "v": torch.randn(B, Hkv, Sk, Dv, generator=g).to(td),
    }
    if dout:
        out["do"] = torch.randn(B, H, Sq, Dv, generator=g).to(td)
    if bias:
        out["key_bias"] = torch.randn(B, H, Sk, generator=g)
    return out


def make_device_inputs(B, H, Sq, Sk, Dqk, Dv, dtype="bf16", seed=42, device="cuda",
                       dout=True, Hkv=None):
    """Same recipe drawn by a CUDA generator, for inputs too large to build on
    the host (the 65536-key decode workload holds 34 GB of K/V)."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    td = DTYPES[dtype]
    Hkv = H if Hkv is None else Hkv
    out = {}
    for name, shape in (("q", (B, H, Sq, Dqk)), ("k", (B, Hkv, Sk, Dqk)), ("v", (B, Hkv, Sk, Dv))):
        t = torch.empty(shape, dtype=td, device=device)
        # draw in fp32 slices so the peak extra memory stays small
        flat = t.view(-1, shape[-1])
        step = 1 << 20
        for r0 in range(0, flat.shape[0], step):
            r1 = min(flat.shape[0], r0 + step)
            flat[r0:r1].copy_(torch.randn(r1 - r0, shape[-1], generator=g, device=device))
        out[name] = t
    if dout:
        out["do"] = torch.randn(B, H, Sq, Dv, generator=g, device=device).to(td)
    return out
