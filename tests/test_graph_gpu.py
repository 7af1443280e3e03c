"""CUDA-graph capture of whole DCP steps.

The entry points only enqueue kernels on the caller's stream: no allocation,
no synchronisation, no host read of device memory.  So a step can be
captured once and replayed: the MLA-decode pack + combine over the exchanged
views, the interleaved pack + fused unpack+combine, the decode attention with
its workspace (the CUDA-core kernel, and the grouped-query tcgen05 kernel with
its split merge), and the absorbed-MLA attention (persistent CTA pairs, with
and without splits).  Replays must reproduce the eager outputs bit for bit,
also after new input values are written into the captured buffers.
"""
import math

import pytest
import torch

from decode_context_attention_gb300 import binding, build, layouts
from decode_context_attention_gb300.workloads import (WORKLOADS, generate, generate_attention,
                                                     generate_mla_attention, scaled)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()


def capture(step):
    """Run `step` once eagerly on a side stream, then capture it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


def same_bytes(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def test_peer_inside_pack_and_combine_replay():
    w = scaled(WORKLOADS["mla_decode"], B=16, seed=71)
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]
    S, B, H, D = o.shape
    N, H_pr = w.N, w.H_pr
    partial_o, stats = layouts.alloc_peer_inside(S, B, H_pr, N, D, o.dtype, DEV)
    dst_o, dst_lse = layouts.peer_inside_send_views(partial_o, stats)
    ro, rl = layouts.exchange_peer_inside(partial_o, stats)
    out = torch.empty((N, B, H_pr, D), dtype=o.dtype, device=DEV)
    out_lse = torch.empty((N, B, H_pr), device=DEV)

    def step():
        binding.pack_send(o, lse, dst_o, dst_lse)
        binding.lse_combine(ro, rl, out, out_lse, base=w.base)

    g = capture(step)
    for seed in (72, 73):
        d2 = generate(scaled(w, seed=seed), DEV)
        o.copy_(d2["o"])
        lse.copy_(d2["lse"])
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        got, got_lse = out.clone(), out_lse.clone()
        step()
        torch.cuda.synchronize()
        assert same_bytes(got, out) and same_bytes(got_lse, out_lse)


def test_interleaved_pack_and_fused_unpack_combine_replay():
    w = scaled(WORKLOADS["mha_decode"], seed=74)
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]
    S, B, H, D = o.shape
    N, H_pr = w.N, w.H_pr
    send = layouts.alloc_peer_major(S, N, B, H_pr, D, o.dtype, DEV)
    pay, words = layouts.peer_major_views(send, D)
    recv = layouts.exchange_peer_major(send)
    out = torch.empty((N, B, H_pr, D), dtype=o.dtype, device=DEV)
    out_lse = torch.empty((N, B, H_pr), device=DEV)

    def step():
        binding.pack_send(o, lse, pay, words)
        binding.unpack_combine(recv, D, out, out_lse, base=w.base)

    g = capture(step)
    o.copy_(generate(scaled(w, seed=75), DEV)["o"])
    g.replay()
    torch.cuda.synchronize()
    got, got_lse = out.clone(), out_lse.clone()
    step()
    torch.cuda.synchronize()
    assert same_bytes(got, out) and same_bytes(got_lse, out_lse)


def test_decode_attention_with_workspace_replay():
    a = generate_attention(B=6, max_len=3000, seed=76)
    c = a["cfg"]
    N, B, H, D = c["N"], c["B"], c["H"], c["D"]
    o = torch.empty((N, B, H, D), dtype=a["q"].dtype, device=DEV)
    lse = torch.empty((N, B, H), device=DEV)
    split = 128
    ws = torch.empty(binding.workspace_bytes(N, B, H, D, a["max_len"], split), dtype=torch.uint8, device=DEV)

    def step():
        binding.decode_attention(a["q"], a["k"], a["v"], a["seq_lens"], a["max_len"], o, lse,
                                 1.0 / math.sqrt(D), base="e", split_tokens=split, workspace=ws)

    g = capture(step)
    a["q"].copy_(torch.randn_like(a["q"], dtype=torch.float32).to(a["q"].dtype))
    a["seq_lens"].copy_(torch.randint(1, a["max_len"] + 1, (B,), device=DEV, dtype=torch.int32))
    g.replay()
    torch.cuda.synchronize()
    got, got_lse = o.clone(), lse.clone()
    step()
    torch.cuda.synchronize()
    assert same_bytes(got, o) and same_bytes(got_lse, lse)


def test_gqa_tensor_core_attention_with_split_merge_replay():
    a = generate_attention("gqa_decode_attention", B=5, max_len=5000, seed=78)
    c = a["cfg"]
    N, B, H, D = c["N"], c["B"], c["H"], c["D"]
    o = torch.empty((N, B, H, D), dtype=a["q"].dtype, device=DEV)
    lse = torch.empty((N, B, H), device=DEV)
    split = 256  # several splits per rank: the tcgen05 kernel and the split merge
    ws = torch.empty(binding.workspace_bytes(N, B, H, D, a["max_len"], split), dtype=torch.uint8, device=DEV)

    def step():
        binding.decode_attention(a["q"], a["k"], a["v"], a["seq_lens"], a["max_len"], o, lse,
                                 1.0 / math.sqrt(D), base="2", split_tokens=split, workspace=ws)

    g = capture(step)
    a["q"].copy_(torch.randn_like(a["q"], dtype=torch.float32).to(a["q"].dtype))
    a["seq_lens"].copy_(torch.randint(0, a["max_len"] + 1, (B,), device=DEV, dtype=torch.int32))
    g.replay()
    torch.cuda.synchronize()
    got, got_lse = o.clone(), lse.clone()
    step()
    torch.cuda.synchronize()
    assert same_bytes(got, o) and same_bytes(got_lse, lse)
    assert binding.device_status() == 0


@pytest.mark.parametrize("split", [512, 4096])
def test_mla_attention_replay(split):
    """The persistent MLA kernel under replay: the item order it makes from
    the lengths on the device follows new lengths written into the captured
    buffer (several splits: the split merge is captured too)."""
    a = generate_mla_attention(B=7, max_len=6000, seed=79)
    c = a["cfg"]
    N, B, H, Dv = c["N"], c["B"], c["H"], c["Dv"]
    o = torch.empty((N, B, H, Dv), dtype=a["q"].dtype, device=DEV)
    lse = torch.empty((N, B, H), device=DEV)
    need = binding.workspace_bytes(N, B, H, Dv, a["max_len"], split)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)

    def step():
        binding.decode_attention_mla(a["q"], a["kv"], a["seq_lens"], a["max_len"], o, lse, c["sm_scale"],
                                     base="2", split_tokens=split, workspace=ws if need else None)

    g = capture(step)
    a["q"].copy_(torch.randn_like(a["q"], dtype=torch.float32).to(a["q"].dtype))
    new_lens = torch.randint(0, a["max_len"] + 1, (B,), device=DEV, dtype=torch.int32)
    new_lens[0] = 0
    a["seq_lens"].copy_(new_lens)
    g.replay()
    torch.cuda.synchronize()
    got, got_lse = o.clone(), lse.clone()
    step()
    torch.cuda.synchronize()
    assert same_bytes(got, o) and same_bytes(got_lse, lse)
    assert binding.device_status() == 0
