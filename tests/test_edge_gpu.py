"""GPU edge cases against the oracle: one rank (identity, bit-exact), empty and
all-empty rows, NaN/+-inf LSE and O with and without sanitising, rank counts
off the fast paths (3, 5, 16, 33), odd head counts and head dims (the 4- and
2-byte vector paths), views that are not 16-byte aligned, G/B = 0, in-place
with several groups, and guard bands around every output."""
import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build, layouts

from parity import (ORACLE_DT, NP_PAYLOAD, assert_bytes_equal, assert_lse_close,
                    assert_merge_close, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.float32, torch.float16, torch.bfloat16]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


def rand_case(G, N, B, Hc, D, dtype, seed, lo=-5.0, hi=5.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    o = torch.randn((G, N, B, Hc, D), generator=g, device=DEV, dtype=torch.float32).to(dtype)
    lse = torch.empty((G, N, B, Hc), device=DEV).uniform_(lo, hi, generator=g)
    return o, lse


class Guarded:
    """An output tensor inside a sentinel-filled buffer with `pad` elements on each side."""

    def __init__(self, shape, dtype, pad=37):
        n = int(np.prod(shape))
        self.pad = pad
        self.buf = torch.empty(n + 2 * pad, dtype=dtype, device=DEV)
        self.buf.view(torch.uint8).fill_(0xA7)
        self.t = self.buf[pad:pad + n].view(shape)

    def check(self):
        b = self.buf.view(torch.uint8).cpu().numpy()
        e = self.buf.element_size()
        assert (b[:self.pad * e] == 0xA7).all() and (b[-self.pad * e:] == 0xA7).all(), "guard band written"


def combine_vs_oracle(o, lse, base="e", sanitize=False, out_shape=None):
    G, N, B, Hc, D = o.shape
    out = Guarded((G, B, Hc, D), o.dtype)
    out_lse = Guarded((G, B, Hc), torch.float32)
    binding.lse_combine(o, lse, out.t, out_lse.t, base=base, sanitize=sanitize)
    want, want_lse = oracle.combine(ORACLE_DT[o.dtype], to_np(o), to_np(lse), base=base,
                                    sanitize=sanitize)
    torch.cuda.synchronize()
    out.check()
    out_lse.check()
    assert_merge_close(out.t, want)
    assert_lse_close(out_lse.t, want_lse)
    return out.t, out_lse.t


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_rank_is_bit_exact_identity(dtype):
    o, lse = rand_case(2, 1, 3, 5, 24, dtype, 1)
    o[0, 0, 0, 0, :3] = torch.tensor([float("nan"), float("inf"), -float("inf")]).to(dtype)
    lse[0, 0, 0, 1] = -float("inf")
    lse[1, 0, 2, 2] = float("nan")
    out = torch.empty((2, 3, 5, 24), dtype=dtype, device=DEV)
    out_lse = torch.empty((2, 3, 5), device=DEV)
    for sanitize in (False, True):
        binding.lse_combine(o, lse, out, out_lse, sanitize=sanitize)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.uint8), o[:, 0].contiguous().view(torch.uint8))
        assert torch.equal(out_lse.view(torch.int32), lse[:, 0].contiguous().view(torch.int32))
    # fused unpack+combine with one rank
    lpd = 4 // o.element_size()
    recv = torch.zeros((2, 1, 3, 5, 24 + lpd), dtype=dtype, device=DEV)
    pay, words = layouts.peer_major_views(recv, 24)
    pay.copy_(o)
    words.copy_(lse)
    binding.unpack_combine(recv, 24, out, out_lse)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), o[:, 0].contiguous().view(torch.uint8))
    assert torch.equal(out_lse.view(torch.int32), lse[:, 0].contiguous().view(torch.int32))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("base", ["e", "2"])
def test_non_finite_lse_classes_and_empty_rows(dtype, base):
    o, lse = rand_case(1, 4, 6, 3, 40, dtype, 2)
    lse[0, :, 0, 0] = -float("inf")                    # all ranks empty
    lse[0, 1, 1, 0] = float("nan")                     # NaN on one rank
    lse[0, 2, 2, 1] = float("inf")                     # +inf on one rank
    lse[0, 0, 3, 2] = float("inf")
    lse[0, 3, 3, 2] = float("nan")                     # NaN and +inf
    lse[0, 0, 4, :] = -float("inf")                    # one empty rank
    o[0, 0, 4, :] = 0
    out, out_lse = combine_vs_oracle(o, lse, base=base)
    assert out_lse[0, 0, 0].item() == -float("inf") and bool((out[0, 0, 0] == 0).all())
    assert np.isnan(out_lse[0, 1, 0].item()) and bool((out[0, 1, 0] == 0).all())


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("sanitize", [False, True])
def test_non_finite_payload(dtype, sanitize):
    o, lse = rand_case(1, 3, 4, 4, 32, dtype, 3)
    o[0, 0, 0, 0, 5] = float("nan")
    o[0, 1, 1, 1, 6] = float("inf")
    o[0, 2, 2, 2, 7] = -float("inf")
    lse[0, 1, 3, 3] = -float("inf")
    o[0, 1, 3, 3, 0] = float("nan")  # NaN under a zero weight: 0 * NaN is NaN unless sanitised
    combine_vs_oracle(o, lse, sanitize=sanitize)


@pytest.mark.parametrize("N", [2, 3, 5, 8, 16, 33])
@pytest.mark.parametrize("dtype", DTYPES)
def test_rank_counts(N, dtype):
    o, lse = rand_case(2, N, 3, 5, 64, dtype, 4 + N, lo=0.0, hi=30.0)
    lse[1, N // 2, 1, :] = -float("inf")
    combine_vs_oracle(o, lse, base="2")


@pytest.mark.parametrize("D", [1, 2, 3, 6, 8, 40, 130, 256, 1000])
@pytest.mark.parametrize("dtype", DTYPES)
def test_head_dims(D, dtype):
    o, lse = rand_case(1, 4, 3, 3, D, dtype, 5 + D)
    combine_vs_oracle(o, lse)


@pytest.mark.parametrize("dtype", DTYPES)
def test_unaligned_views(dtype):
    # shift the whole stack by one element: row starts lose 16-byte alignment
    G, N, B, Hc, D = 1, 4, 5, 3, 64
    base = torch.randn(G * N * B * Hc * D + 1, device=DEV).to(dtype)
    o = base[1:].view(G, N, B, Hc, D)
    lse = torch.empty((G, N, B, Hc), device=DEV).uniform_(-3, 3)
    combine_vs_oracle(o, lse)
    # odd row stride: rows D+1 elements apart
    big = torch.randn((G, N, B, Hc, D + 1), device=DEV).to(dtype)
    combine_vs_oracle(big[..., :D], lse)


def test_empty_inputs_are_no_ops():
    o = torch.randn((1, 2, 0, 4, 8), device=DEV)
    lse = torch.zeros((1, 2, 0, 4), device=DEV)
    out = torch.full((1, 0, 4, 8), 3.0, device=DEV)
    binding.lse_combine(o, lse, out, torch.empty((1, 0, 4), device=DEV))
    o = torch.randn((0, 2, 3, 4, 8), device=DEV)
    binding.lse_combine(o, torch.zeros((0, 2, 3, 4), device=DEV), torch.empty((0, 3, 4, 8), device=DEV))
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", DTYPES)
def test_combine_without_return_lse(dtype):
    o, lse = rand_case(1, 4, 4, 4, 64, dtype, 6)
    out = torch.empty((1, 4, 4, 64), dtype=dtype, device=DEV)
    binding.lse_combine(o, lse, out, None)
    want, _ = oracle.combine(ORACLE_DT[dtype], to_np(o), to_np(lse))
    torch.cuda.synchronize()
    assert_merge_close(out, want)


@pytest.mark.parametrize("N", [1, 3, 8])
def test_in_place_groups(N):
    G, B, H, D = 2, 5, 6, 96
    o, lse = rand_case(G, N, B, H, D, torch.float32, 7 + N)
    o[0, 0, 1, 2, 3] = float("nan")
    lse[1, N - 1, 2, 2] = float("inf")
    o_np, l_np = to_np(o), to_np(lse)
    out_lse = torch.empty((G, B, H), device=DEV)
    binding.lse_combine(o, lse, o[:, 0], out_lse, sanitize=True, inplace=True)
    torch.cuda.synchronize()
    if N == 1:
        assert np.array_equal(to_np(o[:, 0]).view(np.uint32), o_np[:, 0].view(np.uint32))
        return
    want, want_lse = oracle.combine("f32", o_np, l_np, sanitize=True)
    assert_merge_close(o[:, 0], want)
    assert_lse_close(out_lse, want_lse)
    # ranks other than 0 are untouched
    assert np.array_equal(to_np(o[:, 1:]).view(np.uint32), o_np[:, 1:].view(np.uint32))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N,B,H,D", [(2, 3, 6, 5), (4, 1, 12, 2), (3, 2, 9, 130), (8, 2, 8, 64)])
def test_pack_odd_shapes_both_layouts(dtype, N, B, H, D):
    lpd = 4 // torch.empty((), dtype=dtype).element_size()
    if D % lpd:
        pytest.skip("interleaved rows need D % lpd == 0")
    H_pr = H // N
    g = torch.Generator(device=DEV).manual_seed(8)
    o = torch.randn((2, B, H, D), generator=g, device=DEV).to(dtype)
    lse = torch.randn((2, B, H), generator=g, device=DEV)
    # interleaved
    send = torch.empty((2, N, B, H_pr, D + lpd), dtype=dtype, device=DEV)
    send.view(torch.uint8).fill_(0x33)
    pay, words = layouts.peer_major_views(send, D)
    binding.pack_send(o, lse, pay, words)
    send_np = np.empty(send.shape, dtype=NP_PAYLOAD[dtype])
    send_np.view(np.uint8)[...] = 0x33
    oracle.pack(ORACLE_DT[dtype], N, to_np(o), to_np(lse), send_np[..., :D],
                send_np.view(np.float32)[..., D // lpd])
    torch.cuda.synchronize()
    assert_bytes_equal(send, send_np, "send")
    # fused unpack+combine on it
    recv = layouts.exchange_peer_major(send)
    out = torch.empty((N, B, H_pr, D), dtype=dtype, device=DEV)
    out_lse = torch.empty((N, B, H_pr), device=DEV)
    binding.unpack_combine(recv, D, out, out_lse)
    want, want_lse = oracle.unpack_combine(ORACLE_DT[dtype], send_np.transpose(1, 0, 2, 3, 4), D)
    torch.cuda.synchronize()
    assert_merge_close(out, want)
    assert_lse_close(out_lse, want_lse)


@pytest.mark.parametrize("dtype", DTYPES)
def test_pack_strided_source_and_padded_destination(dtype):
    """Source O read through a transposed view; destination rows padded."""
    N, B, H, D = 4, 3, 8, 32
    H_pr = H // N
    base = torch.randn((B, 2, H, D), device=DEV).to(dtype)
    o = base.transpose(0, 1)                       # [G=2, B, H, D], strided
    lse = torch.randn((H, B, 2), device=DEV).permute(2, 1, 0)
    lpd = 4 // o.element_size()
    pad = 3 * lpd
    send = torch.empty((2, N, B, H_pr, D + lpd + pad), dtype=dtype, device=DEV)
    send.view(torch.uint8).fill_(0x42)
    words = send.view(torch.float32)
    binding.pack_send(o, lse, send[..., :D], words[..., D // lpd])
    send_np = np.empty(send.shape, dtype=NP_PAYLOAD[dtype])
    send_np.view(np.uint8)[...] = 0x42
    oracle.pack(ORACLE_DT[dtype], N, to_np(base).transpose(1, 0, 2, 3),
                to_np(lse.permute(2, 1, 0)).transpose(2, 1, 0), send_np[..., :D],
                send_np.view(np.float32)[..., D // lpd])
    torch.cuda.synchronize()
    assert_bytes_equal(send, send_np, "padded send")


def test_errors_raise_through_the_binding():
    o = torch.randn((1, 2, 6, 8), device=DEV)
    lse = torch.randn((1, 2, 6), device=DEV)
    dst = torch.empty((1, 4, 2, 1, 8), device=DEV)
    dl = torch.empty((1, 4, 2, 1), device=DEV)
    with pytest.raises(binding.DcpError) as ei:
        binding.pack_send(o, lse, dst, dl)
    assert ei.value.name == "DCP_ERR_HEADS_NOT_DIVISIBLE"
    with pytest.raises(binding.DcpError):
        x = torch.randn((1, 2, 2, 2, 8), device=DEV)
        binding.lse_combine(x, torch.zeros((1, 2, 2, 2), device=DEV), x[:, 0])  # alias, no flag


def test_pinned_host_operands_match_device_operands():
    """Pinned host tensors as operands: the pack reads its inputs and the combine
    writes its result over the host link; the bytes equal the device path's."""
    N, B, H, D = 4, 6, 16, 128
    H_pr = H // N
    g = torch.Generator(device=DEV).manual_seed(9)
    o = torch.randn((N, B, H, D), generator=g, device=DEV).to(torch.bfloat16)
    lse = torch.empty((N, B, H), device=DEV).uniform_(0, 12, generator=g)
    po, st = layouts.alloc_peer_inside(N, B, H_pr, N, D, torch.bfloat16, DEV)
    po2, st2 = layouts.alloc_peer_inside(N, B, H_pr, N, D, torch.bfloat16, DEV)
    binding.pack_send(o, lse, *layouts.peer_inside_send_views(po, st))
    binding.pack_send(o.cpu().pin_memory(), lse.cpu().pin_memory(), *layouts.peer_inside_send_views(po2, st2))
    torch.cuda.synchronize()
    assert torch.equal(po.view(torch.int16), po2.view(torch.int16))
    assert torch.equal(st[..., 0], st2[..., 0])
    out = torch.empty((N, B, H_pr, D), dtype=torch.bfloat16, device=DEV)
    out_lse = torch.empty((N, B, H_pr), device=DEV)
    out_h = torch.empty((N, B, H_pr, D), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((N, B, H_pr)).pin_memory()
    ro, rl = layouts.exchange_peer_inside(po, st)
    binding.lse_combine(ro, rl, out, out_lse)
    binding.lse_combine(ro, rl, out_h, lse_h)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), out_h.view(torch.int16))
    assert torch.equal(out_lse.cpu(), lse_h)
    with pytest.raises(ValueError):
        binding.lse_combine(ro, rl, torch.empty((N, B, H_pr, D), dtype=torch.bfloat16), None)
