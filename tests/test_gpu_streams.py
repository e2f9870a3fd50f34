"""Stream ordering of the C ABI calls: the same forward + backward issued on
the default stream, on a caller's stream, and captured into a CUDA graph and
replayed on new inputs give bit-identical results (every kernel is
deterministic: no atomics). attn_bwd forks its dQ grid onto a second stream
and joins it back; a missing join shows up here as a race with the reads
that follow on the caller's stream, and under capture as a capture error."""
import pytest
import torch

import block_sparse_attention_tma_gb300 as ga
from block_sparse_attention_tma_gb300.synth import make_inputs
from helpers import assert_no_device_error

pytestmark = pytest.mark.gpu


def _step(g, spec, lists, out, ws, stream=None):
    B, H, S, _ = g["q"].shape
    ga.build_block_mask(B, H, S, S, spec, lists, stream=stream)
    ga.attn_fwd(g["q"], g["k"], g["v"], 0.0, spec, lists, o=out["o"], lse=out["lse"], stream=stream)
    ga.attn_bwd(g["q"], g["k"], g["v"], out["o"], g["do"], out["lse"], 0.0, spec, lists, dq=out["dq"],
                dk=out["dk"], dv=out["dv"], workspace=ws, stream=stream)
    # a read on the caller's stream right after the call: must see the dQ grid's result
    out["dq_sum"].copy_(out["dq"].float().sum(dim=(2, 3)))


def _buffers(g):
    B, H, S, Dqk = g["q"].shape
    Dv = g["v"].shape[-1]
    dev = g["q"].device
    return {"o": torch.empty(B, H, S, Dv, dtype=torch.bfloat16, device=dev),
            "lse": torch.empty(B, H, S, dtype=torch.float32, device=dev),
            "dq": torch.empty_like(g["q"]), "dk": torch.empty_like(g["k"]), "dv": torch.empty_like(g["v"]),
            "dq_sum": torch.empty(B, H, dtype=torch.float32, device=dev)}


@pytest.mark.parametrize("kind,ex,D", [("causal", dict(rel_bias_slope=0.01), 64), ("dyn", {}, 64),
                                       ("sliding", dict(window_left=300), 128)])
def test_streams_and_graph_capture(kind, ex, D):
    B, H, S = 1, 4, 1000
    x = make_inputs(B, H, S, S, D, D, "bf16", seed=5, bias=True)
    g = {n: t.cuda() for n, t in x.items()}
    if kind == "dyn":
        spec = ga.MaskSpec(kind=ga.DYNAMIC_TOPK, topk=300, key_bias=g["key_bias"])
    else:
        spec = ga.MaskSpec(kind={"causal": ga.CAUSAL, "sliding": ga.SLIDING}[kind], **ex)
    lists = ga.alloc_block_lists(B, H, S, S, 128, 128)
    ws = torch.empty(ga.attn_bwd_workspace_bytes(torch.bfloat16, B, H, S, S, D, D), dtype=torch.uint8,
                     device="cuda")
    ref = _buffers(g)
    _step(g, spec, lists, ref, ws)
    torch.cuda.synchronize()
    assert_no_device_error()

    # a caller's stream
    s = torch.cuda.Stream()
    got = _buffers(g)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(g, spec, lists, got, ws, stream=s)
    torch.cuda.synchronize()
    assert_no_device_error()
    for n in ref:
        assert torch.equal(ref[n], got[n]), n

    # captured once, replayed on new inputs written into the same tensors
    cap = _buffers(g)
    graph = torch.cuda.CUDAGraph()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=s):
        _step(g, spec, lists, cap, ws)
    x2 = make_inputs(B, H, S, S, D, D, "bf16", seed=6, bias=True)
    for n in g:
        g[n].copy_(x2[n].cuda())
    graph.replay()
    torch.cuda.synchronize()
    assert_no_device_error()
    ref2 = _buffers(g)
    _step(g, spec, lists, ref2, ws)
    torch.cuda.synchronize()
    for n in ref2:
        assert torch.equal(ref2[n], cap[n]), n
    assert not torch.equal(ref2["o"], ref["o"])  # the replay saw the new inputs


@pytest.mark.parametrize("kind,D,gather", [("dyn", 192, True), ("dyn", 192, False), ("dyn", 64, True),
                                           ("causal", 192, True)])
def test_alternating_inputs_are_independent(kind, D, gather):
    # Two inputs of one shape alternate through the same calls: each result
    # must equal its own first result bit for bit. A kernel that read shared
    # memory or TMEM left over from the previous call (which held the other
    # input's data) would differ.
    B, H, S = 1, 4, 1000
    Dv = 128 if D == 192 else D
    runs = []
    for seed in (11, 12):
        x = make_inputs(B, H, S, S, D, Dv, "bf16", seed=seed, bias=True)
        g = {n: t.cuda() for n, t in x.items()}
        if kind == "dyn":
            spec = ga.MaskSpec(kind=ga.DYNAMIC_TOPK, topk=400, key_bias=g["key_bias"])
        else:
            spec = ga.MaskSpec(kind=ga.CAUSAL, rel_bias_slope=0.01)
        lists = ga.alloc_block_lists(B, H, S, S, 128, 128, gather=gather)
        ws = torch.empty(ga.attn_bwd_workspace_bytes(torch.bfloat16, B, H, S, S, D, Dv), dtype=torch.uint8,
                         device="cuda")
        out = _buffers(g)
        _step(g, spec, lists, out, ws)
        runs.append((g, spec, lists, ws, {n: t.clone() for n, t in out.items()}))
    torch.cuda.synchronize()
    assert_no_device_error()
    for it in range(16):
        g, spec, lists, ws, first = runs[it & 1]
        out = _buffers(g)
        for t in out.values():
            t.fill_(float("nan"))
        _step(g, spec, lists, out, ws)
        torch.cuda.synchronize()
        for n in first:
            assert torch.equal(out[n], first[n]), (it, n)
    assert_no_device_error()


@pytest.mark.parametrize("D,kind", [(192, "causal"), (64, "sliding")])
def test_forward_repeated_calls_are_bitwise_identical(D, kind):
    # The forward's softmax warps of a TMEM lane quarter exchange row maxima
    # through shared memory once per tile; 200 calls in a row, outputs
    # refilled with NaN before each, must all equal the first bit for bit (a
    # read of a partner's maximum before it was written would show).
    B, H, S = 1, 8, 2048
    Dv = 128 if D == 192 else D
    x = make_inputs(B, H, S, S, D, Dv, "bf16", seed=21, dout=False)
    g = {n: t.cuda() for n, t in x.items()}
    if kind == "causal":
        spec = ga.MaskSpec(kind=ga.CAUSAL, rel_bias_slope=0.01)
    else:
        spec = ga.MaskSpec(kind=ga.SLIDING, window_left=300)
    lists = ga.alloc_block_lists(B, H, S, S, 128, 256)
    ga.build_block_mask(B, H, S, S, spec, lists)
    o0, l0 = ga.attn_fwd(g["q"], g["k"], g["v"], 0.0, spec, lists)
    o = torch.empty_like(o0)
    lse = torch.empty_like(l0)
    for it in range(200):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        ga.attn_fwd(g["q"], g["k"], g["v"], 0.0, spec, lists, o=o, lse=lse)
        assert torch.equal(o, o0) and torch.equal(lse, l0), it
    assert_no_device_error()
