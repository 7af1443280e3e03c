"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle, on
the seeded workloads (tiny, MHA decode, MLA decode in bf16 and fp8, the
long-context sweep, cached extend), element by element.

Pack / layout outputs: bit-exact over the WHOLE destination allocation (which
starts filled with the same sentinel bytes on both sides, so a stray write
anywhere, e.g. into stats slot 1 or row padding, fails).  Merges: the
tolerances in tests/parity.py.  The oracle builds its own numpy views of the
same bytes; it shares nothing with the CUDA path but the seeded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build, layouts
from decode_context_attention_gb300.workloads import WORKLOADS, generate, scaled, sweep_points

from parity import (ORACLE_DT, NP_PAYLOAD, assert_bytes_equal, assert_lse_close,
                    assert_merge_close, np_sentinel, sentinel_like, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


def lpd_of(dtype):
    return 4 // torch.empty((), dtype=dtype).element_size()


# ---------------------------------------------------------------------------
# peer-major interleaved: pack + (combine | fused unpack+combine)
# ---------------------------------------------------------------------------

def run_peer_major(w, fused: bool, materialize: bool):
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]                     # [S,B,H,D], [S,B,H]; S = N source ranks
    S, B, H, D = o.shape
    N, H_pr, dt = w.N, w.H_pr, o.dtype
    lpd = lpd_of(dt)
    W = D + lpd
    send = sentinel_like((S, N, B, H_pr, W), dt, DEV)
    pay, words = layouts.peer_major_views(send, D)
    binding.pack_send(o, lse, pay, words)

    # oracle pack over its own numpy views of a sentinel buffer
    o_np, l_np = to_np(o), to_np(lse)
    send_np = np_sentinel((S, N, B, H_pr, W), NP_PAYLOAD[dt])
    oracle.pack(ORACLE_DT[dt], N, o_np, l_np, send_np[..., :D],
                send_np.view(np.float32)[..., D // lpd])
    torch.cuda.synchronize()
    assert_bytes_equal(send, send_np, f"{w.name} peer-major send buffer")

    # exchange model: destination d receives send[s, d] from every source s
    recv = layouts.materialize_peer_major(send) if materialize else layouts.exchange_peer_major(send)
    out = torch.empty((N, B, H_pr, D), dtype=dt, device=DEV)
    out_lse = torch.empty((N, B, H_pr), dtype=torch.float32, device=DEV)
    if fused:
        binding.unpack_combine(recv, D, out, out_lse, base=w.base)
    else:
        rp, rw = layouts.peer_major_views(recv, D)
        binding.lse_combine(rp, rw, out, out_lse, base=w.base)
    recv_np = send_np.transpose(1, 0, 2, 3, 4)
    if fused:
        want, want_lse = oracle.unpack_combine(ORACLE_DT[dt], recv_np, D, base=w.base)
    else:
        want, want_lse = oracle.combine(ORACLE_DT[dt], recv_np[..., :D],
                                        recv_np.view(np.float32)[..., D // lpd], base=w.base)
    torch.cuda.synchronize()
    st = assert_merge_close(out, want, f"{w.name} out")
    assert_lse_close(out_lse, want_lse, f"{w.name} out_lse")
    return st


@pytest.mark.parametrize("materialize", [False, True])
def test_tiny_peer_major_pack_and_combine(materialize):
    run_peer_major(WORKLOADS["tiny"], fused=False, materialize=materialize)


@pytest.mark.parametrize("materialize", [False, True])
def test_mha_decode_pack_and_fused_unpack_combine(materialize):
    run_peer_major(WORKLOADS["mha_decode"], fused=True, materialize=materialize)


def test_mha_decode_strided_combine_on_interleaved_views():
    run_peer_major(WORKLOADS["mha_decode"], fused=False, materialize=False)


@pytest.mark.parametrize("materialize", [False, True])
def test_mla_decode_fp8_pack_and_fused_unpack_combine(materialize):
    run_peer_major(WORKLOADS["mla_decode_fp8"], fused=True, materialize=materialize)


def test_mla_decode_fp8_strided_combine_on_interleaved_views():
    run_peer_major(WORKLOADS["mla_decode_fp8"], fused=False, materialize=False)


# ---------------------------------------------------------------------------
# peer-inside split: pack + combine over the strided receive views
# ---------------------------------------------------------------------------

def run_peer_inside(w, materialize: bool, stats_fill: float = -7777.0):
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]
    S, B, H, D = o.shape
    N, H_pr, dt = w.N, w.H_pr, o.dtype
    partial_o = sentinel_like((S, B, H_pr, N, D), dt, DEV)
    stats = torch.full((S, B, H_pr, N, 2), stats_fill, dtype=torch.float32, device=DEV)
    dst_o, dst_lse = layouts.peer_inside_send_views(partial_o, stats)
    binding.pack_send(o, lse, dst_o, dst_lse)

    o_np, l_np = to_np(o), to_np(lse)
    po_np = np_sentinel((S, B, H_pr, N, D), NP_PAYLOAD[dt])
    st_np = np.full((S, B, H_pr, N, 2), stats_fill, dtype=np.float32)
    oracle.pack(ORACLE_DT[dt], N, o_np, l_np, po_np.transpose(0, 3, 1, 2, 4),
                st_np[..., 0].transpose(0, 3, 1, 2))
    torch.cuda.synchronize()
    assert_bytes_equal(partial_o, po_np, f"{w.name} partial_o")
    assert_bytes_equal(stats, st_np, f"{w.name} stats (slot 1 must stay {stats_fill})")

    if materialize:
        ro, rl = layouts.materialize_peer_inside(partial_o, stats)
    else:
        ro, rl = layouts.exchange_peer_inside(partial_o, stats)
    out = torch.empty((N, B, H_pr, D), dtype=dt, device=DEV)
    out_lse = torch.empty((N, B, H_pr), dtype=torch.float32, device=DEV)
    binding.lse_combine(ro, rl, out, out_lse, base=w.base)
    want, want_lse = oracle.combine(ORACLE_DT[dt], po_np.transpose(3, 0, 1, 2, 4),
                                    st_np[..., 0].transpose(3, 0, 1, 2), base=w.base)
    torch.cuda.synchronize()
    st = assert_merge_close(out, want, f"{w.name} out")
    assert_lse_close(out_lse, want_lse, f"{w.name} out_lse")
    return st


@pytest.mark.parametrize("materialize", [False, True])
def test_mla_decode_peer_inside_pack_and_strided_combine(materialize):
    run_peer_inside(WORKLOADS["mla_decode"], materialize=materialize)


@pytest.mark.parametrize("materialize", [False, True])
def test_mla_decode_fp8_peer_inside_pack_and_strided_combine(materialize):
    run_peer_inside(scaled(WORKLOADS["mla_decode_fp8"], B=32, layout="peer_inside", seed=61),
                    materialize=materialize)


def test_page_peer_inside_shapes_with_zero_stats():
    """sglang PR #34651's own layout test shapes (N,B,H_pr,D) = (2,4,8,128), (4,1,16,512),
    bf16, stats initialised to zero: slot 1 must stay zero."""
    for N, B, H_pr, D in ((2, 4, 8, 128), (4, 1, 16, 512)):
        w = scaled(WORKLOADS["mla_decode"], N=N, B=B, H=H_pr * N, D=D, base="e", seed=11 + N)
        run_peer_inside(w, materialize=False, stats_fill=0.0)


def _page_case(key):
    import json
    import os
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_cases.json")) as f:
        return json.load(f)[key]["value"]


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("layout", ["peer_major", "peer_inside"])
def test_bf16_error_within_what_the_pages_observed(N, layout):
    """At the shape sglang PR #34651 quotes its bf16 error for (B=8, 12 heads per
    rank, D=512; the rank count is not given, so 2, 4 and 8), the merged bf16
    output's largest error relative to the fp64 oracle stays below the 7.8e-3
    the page reports against its fp32 reference, and below the 3e-2 that vLLM
    PR #41160's half-precision test allows."""
    w = scaled(WORKLOADS["mla_decode"], N=N, B=8, H=12 * N, D=512, layout=layout, seed=80 + N)
    st = run_peer_major(w, fused=True, materialize=False) if layout == "peer_major" \
        else run_peer_inside(w, materialize=False)
    assert st["rel"] <= _page_case("bf16_merge_error_observed")
    assert st["rel"] <= _page_case("half_precision_test_rtol")


# ---------------------------------------------------------------------------
# long-context decode sweep: 48 points, both layouts
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", sweep_points(), ids=lambda w: w.name)
def test_sweep_point(w):
    if w.layout == "peer_major":
        run_peer_major(w, fused=True, materialize=False)
    else:
        run_peer_inside(w, materialize=False)


@pytest.mark.parametrize("N,B,D", [(2, 8, 128), (8, 256, 512)])
def test_two_collective_layout(N, B, D):
    """The legacy layout: O and LSE packed into separate peer-major buffers (one
    all-to-all each), then the combine over the exchanged views without a
    returned LSE.  The sweep recipe; the second case is its largest point."""
    w = [p for p in sweep_points() if p.layout == "peer_major" and p.N == N and p.B == B and p.D == D][0]
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]
    S, _, H, _ = o.shape
    H_pr, dt = w.H_pr, o.dtype
    send_o = sentinel_like((S, N, B, H_pr, D), dt, DEV)
    send_l = sentinel_like((S, N, B, H_pr), torch.float32, DEV)
    binding.pack_send(o, lse, send_o, send_l)
    so_np = np_sentinel((S, N, B, H_pr, D), NP_PAYLOAD[dt])
    sl_np = np_sentinel((S, N, B, H_pr), np.float32)
    oracle.pack(ORACLE_DT[dt], N, to_np(o), to_np(lse), so_np, sl_np)
    torch.cuda.synchronize()
    assert_bytes_equal(send_o, so_np, "separate O send buffer")
    assert_bytes_equal(send_l, sl_np, "separate LSE send buffer")
    out = torch.empty((N, B, H_pr, D), dtype=dt, device=DEV)
    binding.lse_combine(send_o.transpose(0, 1), send_l.transpose(0, 1), out, None, base=w.base)
    want, _ = oracle.combine(ORACLE_DT[dt], so_np.transpose(1, 0, 2, 3, 4), sl_np.transpose(1, 0, 2, 3),
                             base=w.base)
    torch.cuda.synchronize()
    assert_merge_close(out, want, f"{w.name} two-collective out")


# ---------------------------------------------------------------------------
# cached extend: in-place sanitising combine + head slices
# ---------------------------------------------------------------------------

def run_inplace(w, sample: int | None):
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]                       # [N,T,H,D] fp32, [N,T,H]
    N, T, H, D = o.shape
    if sample is None:
        o_np, l_np = to_np(o), to_np(lse)
        rows = None
    else:
        # the rows whose LSE has an injected NaN/inf, plus random rows; inputs
        # are gathered before the call overwrites rank 0
        g = torch.Generator(device="cpu").manual_seed(1234)
        special = (~torch.isfinite(lse)).any(dim=0).nonzero().cpu()
        rnd = torch.stack([torch.randint(0, T, (sample,), generator=g),
                           torch.randint(0, H, (sample,), generator=g)], dim=1)
        rows = torch.cat([special, rnd, torch.tensor([[0, 0], [T - 1, H - 1]])]).to(DEV)
        o_np = to_np(o[:, rows[:, 0], rows[:, 1], :])[:, None]   # [N, 1, K, D]
        l_np = to_np(lse[:, rows[:, 0], rows[:, 1]])[:, None]    # [N, 1, K]
    out_lse = torch.empty((T, H), dtype=torch.float32, device=DEV)
    out = o[0]
    binding.lse_combine(o, lse, out, out_lse, base=w.base, sanitize=True, inplace=True)
    want, want_lse = oracle.combine("f32", o_np[None], l_np[None], base=w.base, sanitize=True)
    torch.cuda.synchronize()
    if rows is None:
        assert_merge_close(out, want[0], f"{w.name} out")
        assert_lse_close(out_lse, want_lse[0], f"{w.name} out_lse")
    else:
        assert_merge_close(out[rows[:, 0], rows[:, 1]], want[0, 0], f"{w.name} sampled out")
        assert_lse_close(out_lse[rows[:, 0], rows[:, 1]], want_lse[0, 0], f"{w.name} sampled lse")
        # properties over every row: sanitised output is finite; the global LSE
        # is NaN exactly where some rank's LSE is NaN
        assert bool(torch.isfinite(out).all())
        assert torch.equal(torch.isnan(out_lse), torch.isnan(lse).any(dim=0))
    # head slices are views: rank k keeps heads [k*H/N, (k+1)*H/N)
    hs = H // N
    for k in range(N):
        sl = out[:, k * hs:(k + 1) * hs, :]
        assert sl.data_ptr() == out.data_ptr() + k * hs * D * out.element_size()
        assert out_lse[:, k * hs:(k + 1) * hs].shape == (T, hs)


def test_cached_extend_small_all_rows():
    run_inplace(scaled(WORKLOADS["cached_extend"], B=48, seed=41), sample=None)


def test_cached_extend_full_size_sampled():
    """16384 x 96 x 512 fp32 per rank, 8 ranks (24 GiB), the launch the benchmark times."""
    run_inplace(WORKLOADS["cached_extend"], sample=4096)


def test_cached_extend_contiguous_head_slices_in_one_launch():
    """The ag_rs merge's per-rank head slices (rank k keeps heads [k*H/N, (k+1)*H/N),
    made contiguous) produced directly by the combine's store: the group axis
    walks the slices, so one launch writes out[k] = merged heads of slice k as a
    contiguous [T, H/N, D] block.  Compared with the oracle and, bit for bit,
    with the slices of the in-place result."""
    w = scaled(WORKLOADS["cached_extend"], B=40, seed=43)
    d = generate(w, DEV)
    o, lse = d["o"], d["lse"]                     # [N, T, H, D], [N, T, H]
    N, T, H, D = o.shape
    hs = H // N
    o_np, l_np = to_np(o), to_np(lse)
    o_k = o.view(N, T, N, hs, D).permute(2, 0, 1, 3, 4)     # [slice k][rank][T][hs][D]
    l_k = lse.view(N, T, N, hs).permute(2, 0, 1, 3)
    slices = torch.empty((N, T, hs, D), dtype=o.dtype, device=DEV)
    slices_lse = torch.empty((N, T, hs), dtype=torch.float32, device=DEV)
    binding.lse_combine(o_k, l_k, slices, slices_lse, base=w.base, sanitize=True)
    want, want_lse = oracle.combine("f32", o_np[None], l_np[None], base=w.base, sanitize=True)
    torch.cuda.synchronize()
    want_k = want[0].reshape(T, N, hs, D).transpose(1, 0, 2, 3)
    want_lk = want_lse[0].reshape(T, N, hs).transpose(1, 0, 2)
    assert_merge_close(slices, want_k, "contiguous slices")
    assert_lse_close(slices_lse, want_lk, "contiguous slice lse")
    # the in-place merge, sliced afterwards, holds the same bytes
    out_lse = torch.empty((T, H), dtype=torch.float32, device=DEV)
    binding.lse_combine(o, lse, o[0], out_lse, base=w.base, sanitize=True, inplace=True)
    torch.cuda.synchronize()
    for k in range(N):
        assert torch.equal(slices[k].view(torch.int32), o[0][:, k * hs:(k + 1) * hs].contiguous().view(torch.int32))
        assert torch.equal(slices_lse[k].view(torch.int32),
                           out_lse[:, k * hs:(k + 1) * hs].contiguous().view(torch.int32))
