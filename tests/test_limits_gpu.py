"""The largest sizes the library accepts, against the oracle: N = 4096 ranks
(the ABI's maximum) through the pack (4096 peers, and 4096 source groups),
the fused unpack+combine over 4096 interleaved rows per output row and the
strided combine over 4096 partials (the any-N merge kernel), and payload rows
far longer than any workload's (64 KiB and more per row, the generic merge
path that walks a row in several passes)."""
import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build, layouts

from parity import (NP_PAYLOAD, ORACLE_DT, assert_bytes_equal, assert_lse_close,
                    assert_merge_close, np_sentinel, sentinel_like, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8 = torch.float8_e4m3fn
DTYPES = [torch.float32, torch.float16, torch.bfloat16, FP8]
N_MAX = 4096


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


def lpd_of(dtype):
    return 4 // torch.empty((), dtype=dtype).element_size()


def payload(shape, dtype, g):
    x = torch.randn(shape, generator=g, device=DEV)
    return x.clamp(-440, 440).to(dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_pack_to_the_largest_peer_count(dtype):
    """N = 4096 peers, H = 4096 heads: one head per peer, both send layouts."""
    N, B, D = N_MAX, 2, 40
    lpd = lpd_of(dtype)
    g = torch.Generator(device=DEV).manual_seed(4096)
    o = payload((1, B, N, D), dtype, g)
    lse = torch.empty((1, B, N), device=DEV).uniform_(-20, 20, generator=g)
    o_np, l_np = to_np(o), to_np(lse)
    # peer-major interleaved [N, B, 1, D + lpd]
    send = sentinel_like((1, N, B, 1, D + lpd), dtype, DEV, 0x33)
    binding.pack_send(o, lse, *layouts.peer_major_views(send, D))
    want = np_sentinel(send.shape, NP_PAYLOAD[dtype], 0x33)
    oracle.pack(ORACLE_DT[dtype], N, o_np, l_np, want[..., :D], want.view(np.float32)[..., D // lpd])
    # peer-inside split: O [B, 1, N, D], stats [B, 1, N, 2] (slot 1 untouched)
    po, st = layouts.alloc_peer_inside(1, B, 1, N, D, dtype, DEV)
    po.view(torch.uint8).fill_(0x44)
    st.view(torch.uint8).fill_(0x55)
    binding.pack_send(o, lse, *layouts.peer_inside_send_views(po, st))
    want_po = np_sentinel(po.shape, NP_PAYLOAD[dtype], 0x44)
    want_st = np_sentinel(st.shape, np.float32, 0x55)
    oracle.pack(ORACLE_DT[dtype], N, o_np, l_np, want_po.transpose(0, 3, 1, 2, 4),
                want_st[..., 0].transpose(0, 3, 1, 2))
    torch.cuda.synchronize()
    assert_bytes_equal(send, want, "interleaved send, N = 4096")
    assert_bytes_equal(po, want_po, "peer-inside partial_o, N = 4096")
    assert_bytes_equal(st, want_st, "peer-inside stats, N = 4096")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("base", ["e", "2"])
def test_merges_over_the_largest_rank_count(dtype, base):
    """4096 source groups packed into interleaved rows for one peer, then merged
    over all 4096 of them: fused unpack+combine, and the strided combine over
    the payload / LSE-word views of the same rows."""
    S, B, H, D = N_MAX, 2, 3, 40
    lpd = lpd_of(dtype)
    g = torch.Generator(device=DEV).manual_seed(4097)
    o = payload((S, B, H, D), dtype, g)
    lse = torch.empty((S, B, H), device=DEV).uniform_(0, 30, generator=g)
    lse[::7, 1, 2] = -float("inf")          # ranks that own no KV for one row
    lse[:, 0, 1] = -float("inf")            # a row no rank owns: out 0, lse -inf
    send = sentinel_like((S, 1, B, H, D + lpd), dtype, DEV, 0x33)
    binding.pack_send(o, lse, *layouts.peer_major_views(send, D))
    recv = layouts.exchange_peer_major(send)          # [1, S, B, H, D + lpd]
    out = sentinel_like((1, B, H, D), dtype, DEV)
    out_lse = sentinel_like((1, B, H), torch.float32, DEV)
    binding.unpack_combine(recv, D, out, out_lse, base=base)
    send_np = np_sentinel(send.shape, NP_PAYLOAD[dtype], 0x33)
    oracle.pack(ORACLE_DT[dtype], 1, to_np(o), to_np(lse), send_np[..., :D],
                send_np.view(np.float32)[..., D // lpd])
    want, want_lse = oracle.unpack_combine(ORACLE_DT[dtype], send_np.transpose(1, 0, 2, 3, 4), D, base=base)
    # the same merge through strided views of the payload and the LSE words
    pay, words = layouts.peer_major_views(recv, D)
    out2 = sentinel_like((1, B, H, D), dtype, DEV)
    out2_lse = sentinel_like((1, B, H), torch.float32, DEV)
    binding.lse_combine(pay, words, out2, out2_lse, base=base)
    torch.cuda.synchronize()
    assert_bytes_equal(send, send_np, "send of 4096 groups")
    for got, got_lse in ((out, out_lse), (out2, out2_lse)):
        assert_merge_close(got, want)
        assert_lse_close(got_lse, want_lse)
    assert float(want_lse[0, 0, 1]) == -np.inf and not np.any(want[0, 0, 1].astype(np.float64))


@pytest.mark.parametrize("dtype,D", [(torch.float32, 16384), (torch.float16, 32768),
                                     (torch.bfloat16, 32768), (FP8, 65536), (torch.float32, 16383),
                                     (torch.bfloat16, 32762)])
def test_long_rows(dtype, D):
    """Rows of 64 KiB (and ragged lengths just below) through the combine and,
    where D is a multiple of lpd, the interleaved pack and fused unpack+combine."""
    N, B, H = 3, 2, 2
    g = torch.Generator(device=DEV).manual_seed(D)
    o = payload((N, B, H, D), dtype, g)
    lse = torch.empty((N, B, H), device=DEV).uniform_(-5, 5, generator=g)
    out = sentinel_like((1, B, H, D), dtype, DEV)
    out_lse = sentinel_like((1, B, H), torch.float32, DEV)
    binding.lse_combine(o.unsqueeze(0), lse.unsqueeze(0), out, out_lse, base="2")
    want, want_lse = oracle.combine(ORACLE_DT[dtype], to_np(o)[None], to_np(lse)[None], base="2")
    torch.cuda.synchronize()
    assert_merge_close(out, want)
    assert_lse_close(out_lse, want_lse)
    lpd = lpd_of(dtype)
    if D % lpd:
        return
    send = sentinel_like((N, 1, B, H, D + lpd), dtype, DEV, 0x33)
    binding.pack_send(o, lse, *layouts.peer_major_views(send, D))
    out3 = sentinel_like((1, B, H, D), dtype, DEV)
    binding.unpack_combine(layouts.exchange_peer_major(send), D, out3, None, base="2")
    torch.cuda.synchronize()
    assert_merge_close(out3, want)
