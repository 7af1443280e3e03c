"""fp8 e4m3 payloads against the oracle: the pack bit for bit (both send
layouts, lpd = 4 in the interleaved rows), merges within half an e4m3 ulp
(tests/parity.py), one rank as a bit-exact identity, NaN payload bytes with
and without sanitising, non-finite LSE classes, rank counts off the fast
paths, head dims from 4 to 2048, magnitudes up to the e4m3 maximum, views
that are 4- but not 16-byte aligned, and a seeded random sweep over storage
orders.  Views that break the 4-byte row granularity must be refused."""
import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build, layouts

from parity import assert_bytes_equal, assert_lse_close, assert_merge_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8 = torch.float8_e4m3fn
NAN8 = 0x7F     # S.1111.111: the e4m3 NaN


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


def fp8_case(G, N, B, Hc, D, seed, scale=1.0, lo=-5.0, hi=5.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    o = (torch.randn((G, N, B, Hc, D), generator=g, device=DEV) * scale).clamp(-440, 440).to(FP8)
    lse = torch.empty((G, N, B, Hc), device=DEV).uniform_(lo, hi, generator=g)
    return o, lse


def set_nan(o, idx):
    o.view(torch.uint8)[idx] = NAN8


def guarded(shape, dtype, pad=40):
    """(buffer with sentinel guard bands, the output view inside it); the pad
    keeps fp8 rows on the 4-byte grid."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * pad, dtype=dtype, device=DEV)
    buf.view(torch.uint8).fill_(0xA7)
    return buf, buf[pad:pad + n].view(shape)


def check_guards(buf, pad=40):
    b = buf.view(torch.uint8).cpu().numpy()
    e = buf.element_size()
    assert (b[:pad * e] == 0xA7).all() and (b[-pad * e:] == 0xA7).all(), "guard band written"


def combine_vs_oracle(o, lse, base="e", sanitize=False):
    G, N, B, Hc, D = o.shape
    ob, out = guarded((G, B, Hc, D), FP8)
    lb, out_lse = guarded((G, B, Hc), torch.float32)
    binding.lse_combine(o, lse, out, out_lse, base=base, sanitize=sanitize)
    want, want_lse = oracle.combine("fp8", to_np(o), to_np(lse), base=base, sanitize=sanitize)
    torch.cuda.synchronize()
    check_guards(ob)
    check_guards(lb)
    assert_merge_close(out, want)
    assert_lse_close(out_lse, want_lse)
    return out, out_lse, want


def test_single_rank_is_bit_exact_identity():
    o, lse = fp8_case(2, 1, 3, 5, 24, 1)
    set_nan(o, (0, 0, 0, 0, slice(0, 3)))
    lse[0, 0, 0, 1] = -float("inf")
    lse[1, 0, 2, 2] = float("nan")
    out = torch.empty((2, 3, 5, 24), dtype=FP8, device=DEV)
    out_lse = torch.empty((2, 3, 5), device=DEV)
    for sanitize in (False, True):
        binding.lse_combine(o, lse, out, out_lse, sanitize=sanitize)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.uint8), o[:, 0].contiguous().view(torch.uint8))
        assert torch.equal(out_lse.view(torch.int32), lse[:, 0].contiguous().view(torch.int32))
    recv = torch.zeros((2, 1, 3, 5, 24 + 4), dtype=FP8, device=DEV)
    pay, words = layouts.peer_major_views(recv, 24)
    pay.copy_(o)
    words.copy_(lse)
    binding.unpack_combine(recv, 24, out, out_lse)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), o[:, 0].contiguous().view(torch.uint8))
    assert torch.equal(out_lse.view(torch.int32), lse[:, 0].contiguous().view(torch.int32))


@pytest.mark.parametrize("base", ["e", "2"])
def test_non_finite_lse_classes_and_empty_rows(base):
    o, lse = fp8_case(1, 4, 6, 3, 40, 2)
    lse[0, :, 0, 0] = -float("inf")                    # all ranks empty
    lse[0, 1, 1, 0] = float("nan")
    lse[0, 2, 2, 1] = float("inf")
    lse[0, 0, 3, 2] = float("inf")
    lse[0, 3, 3, 2] = float("nan")
    lse[0, 0, 4, :] = -float("inf")                    # one empty rank
    o.view(torch.uint8)[0, 0, 4] = 0
    out, out_lse, _ = combine_vs_oracle(o, lse, base=base)
    assert out_lse[0, 0, 0].item() == -float("inf")
    assert bool((out[0, 0, 0].float() == 0).all())


@pytest.mark.parametrize("sanitize", [False, True])
def test_nan_payload(sanitize):
    o, lse = fp8_case(1, 3, 4, 4, 32, 3)
    set_nan(o, (0, 0, 0, 0, 5))
    set_nan(o, (0, 1, 1, 1, 6))
    lse[0, 1, 3, 3] = -float("inf")
    set_nan(o, (0, 1, 3, 3, 0))   # NaN under a zero weight: 0 * NaN is NaN unless sanitised
    out, _, want = combine_vs_oracle(o, lse, sanitize=sanitize)
    assert np.isnan(want).any() != sanitize


@pytest.mark.parametrize("N", [2, 3, 5, 8, 16, 33])
def test_rank_counts(N):
    o, lse = fp8_case(2, N, 3, 5, 64, 4 + N, lo=0.0, hi=30.0)
    lse[1, N // 2, 1, :] = -float("inf")
    combine_vs_oracle(o, lse, base="2")


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("D", [4, 12, 40, 128, 132, 512, 1000, 2048])
def test_head_dims(N, D):
    o, lse = fp8_case(1, N, 3, 3, D, 5 + D + N)
    combine_vs_oracle(o, lse)


def test_magnitudes_up_to_the_e4m3_maximum():
    o, lse = fp8_case(1, 4, 16, 8, 128, 6, scale=200.0)
    o.view(torch.uint8)[0, :, 0, 0, :4] = torch.tensor([0x7E, 0xFE, 0x7E, 0xFE], dtype=torch.uint8,
                                                       device=DEV)  # +-448
    out, _, want = combine_vs_oracle(o, lse)
    assert not np.isnan(want).any()
    assert not torch.isnan(out.float()).any()


def test_four_byte_aligned_views():
    G, N, B, Hc, D = 1, 4, 5, 3, 64
    base = torch.randn(G * N * B * Hc * D + 4, device=DEV).to(FP8)
    lse = torch.empty((G, N, B, Hc), device=DEV).uniform_(-3, 3)
    combine_vs_oracle(base[4:].view(G, N, B, Hc, D), lse)     # starts 4 bytes in
    big = torch.randn((G, N, B, Hc, D + 4), device=DEV).to(FP8)
    combine_vs_oracle(big[..., :D], lse)                       # rows D + 4 bytes apart


def test_rows_off_the_four_byte_grid_are_refused():
    G, N, B, Hc, D = 1, 4, 5, 3, 64
    lse = torch.zeros((G, N, B, Hc), device=DEV)
    out = torch.empty((G, B, Hc, D), dtype=FP8, device=DEV)
    base = torch.zeros(G * N * B * Hc * D + 1, device=DEV).to(FP8)
    with pytest.raises(binding.DcpError) as ei:
        binding.lse_combine(base[1:].view(G, N, B, Hc, D), lse, out)
    assert ei.value.name == "DCP_ERR_MISALIGNED"
    odd = torch.zeros((G, N, B, Hc, 6), device=DEV).to(FP8)
    with pytest.raises(binding.DcpError) as ei:
        binding.lse_combine(odd, lse, torch.empty((G, B, Hc, 6), dtype=FP8, device=DEV))
    assert ei.value.name == "DCP_ERR_MISALIGNED"
    with pytest.raises(binding.DcpError) as ei:
        binding.pack_send(torch.zeros((1, 2, 4, 6), device=DEV).to(FP8), torch.zeros((1, 2, 4), device=DEV),
                          torch.empty((1, 2, 2, 2, 6), dtype=FP8, device=DEV),
                          torch.empty((1, 2, 2, 2), device=DEV))
    assert ei.value.name == "DCP_ERR_MISALIGNED"


def test_combine_without_return_lse():
    o, lse = fp8_case(1, 4, 4, 4, 64, 7)
    out = torch.empty((1, 4, 4, 64), dtype=FP8, device=DEV)
    binding.lse_combine(o, lse, out, None)
    want, _ = oracle.combine("fp8", to_np(o), to_np(lse))
    torch.cuda.synchronize()
    assert_merge_close(out, want)


@pytest.mark.parametrize("N,B,H,D", [(2, 3, 6, 4), (4, 1, 12, 12), (3, 2, 9, 132), (8, 2, 8, 64)])
def test_pack_both_layouts_and_fused_unpack(N, B, H, D):
    H_pr = H // N
    g = torch.Generator(device=DEV).manual_seed(8 + D)
    o = torch.randn((2, B, H, D), generator=g, device=DEV).to(FP8)
    lse = torch.randn((2, B, H), generator=g, device=DEV)
    # interleaved: [payload D bytes | LSE word], lpd = 4
    send = torch.empty((2, N, B, H_pr, D + 4), dtype=FP8, device=DEV)
    send.view(torch.uint8).fill_(0x33)
    pay, words = layouts.peer_major_views(send, D)
    binding.pack_send(o, lse, pay, words)
    send_np = np.full(send.shape, 0x33, dtype=np.uint8)
    oracle.pack("fp8", N, to_np(o), to_np(lse), send_np[..., :D], send_np.view(np.float32)[..., D // 4])
    torch.cuda.synchronize()
    assert_bytes_equal(send, send_np, "send")
    recv = layouts.exchange_peer_major(send)
    out = torch.empty((N, B, H_pr, D), dtype=FP8, device=DEV)
    out_lse = torch.empty((N, B, H_pr), device=DEV)
    binding.unpack_combine(recv, D, out, out_lse)
    want, want_lse = oracle.unpack_combine("fp8", send_np.transpose(1, 0, 2, 3, 4), D)
    torch.cuda.synchronize()
    assert_merge_close(out, want)
    assert_lse_close(out_lse, want_lse)
    # peer-inside split
    po = torch.empty((2, B, H_pr, N, D), dtype=FP8, device=DEV)
    po.view(torch.uint8).fill_(0x3C)
    st = torch.full((2, B, H_pr, N, 2), -3.25, device=DEV)
    binding.pack_send(o, lse, po.permute(0, 3, 1, 2, 4), st[..., 0].permute(0, 3, 1, 2))
    po_np = np.full(po.shape, 0x3C, dtype=np.uint8)
    st_np = np.full(st.shape, -3.25, dtype=np.float32)
    oracle.pack("fp8", N, to_np(o), to_np(lse), po_np.transpose(0, 3, 1, 2, 4),
                st_np[..., 0].transpose(0, 3, 1, 2))
    torch.cuda.synchronize()
    assert_bytes_equal(po, po_np, "partial_o")
    assert_bytes_equal(st, st_np, "stats (slot 1 untouched)")


def strided(shape, rng):
    """An fp8 tensor of `shape` with its outer axes stored in a random order and
    its start 0, 4 or 8 bytes into the buffer (row starts stay 4-byte aligned
    when the last axis is a multiple of 4)."""
    nd = len(shape)
    order = list(rng.permutation(nd - 1)) + [nd - 1]
    store = [shape[i] for i in order]
    off = 4 * int(rng.integers(0, 3))
    n = int(np.prod(store))
    buf = torch.empty(n + off, dtype=FP8, device=DEV)
    t = buf[off:off + n].view(store)
    return t.permute(*[order.index(i) for i in range(nd)])


@pytest.mark.parametrize("seed", range(20))
def test_random_combine(seed):
    rng = np.random.default_rng(5000 + seed)
    N = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 16, 33]))
    G, B, Hc = int(rng.integers(1, 4)), int(rng.integers(1, 7)), int(rng.integers(1, 10))
    D = 4 * int(rng.choice([1, 2, 3, 16, 25, 32, 64, 128, 150]))
    base = str(rng.choice(["e", "2"]))
    sanitize = bool(rng.integers(2))
    g = torch.Generator(device=DEV).manual_seed(int(rng.integers(1 << 30)))
    o = strided((G, N, B, Hc, D), rng)
    o.copy_(torch.randn(o.shape, generator=g, device=DEV).to(FP8))
    lse = torch.empty((G, N, B, Hc), device=DEV).uniform_(-10, 25, generator=g)
    if rng.integers(2):
        lse[0, 0, 0, 0] = -float("inf")
        set_nan(o, tuple(int(rng.integers(n)) for n in o.shape))
    out = strided((G, B, Hc, D), rng)
    out_lse = torch.empty((G, B, Hc), device=DEV)
    binding.lse_combine(o, lse, out, out_lse, base=base, sanitize=sanitize)
    want, want_lse = oracle.combine("fp8", to_np(o), to_np(lse), base=base, sanitize=sanitize)
    torch.cuda.synchronize()
    if N == 1:
        assert torch.equal(out.contiguous().view(torch.uint8), o[:, 0].contiguous().view(torch.uint8))
    else:
        assert_merge_close(out, want)
    assert_lse_close(out_lse, want_lse)
