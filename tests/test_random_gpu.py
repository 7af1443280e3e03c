"""Seeded randomized parity sweep: pack, combine and fused unpack+combine on
random shapes, payload types, LSE bases, flags and storage orders (random
axis permutations, element offsets that break 16-byte alignment, padded
interleaved rows), against the fp64 oracle.  Pack outputs are compared bit
for bit over the whole destination buffer; merges with tests/parity.py's
tolerances."""
import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build

from parity import (NP_PAYLOAD, ORACLE_DT, assert_bytes_equal, assert_lse_close, assert_merge_close,
                    to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"
TYPES = [torch.float32, torch.float16, torch.bfloat16]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


def strided(shape, dtype, rng, offset_max=3):
    """A tensor of `shape` whose outer axes are stored in a random order, last
    axis innermost, starting `off` elements into its buffer."""
    nd = len(shape)
    order = list(rng.permutation(nd - 1)) + [nd - 1]
    store = [shape[i] for i in order]
    off = int(rng.integers(0, offset_max + 1))
    n = int(np.prod(store))
    buf = torch.empty(n + off, dtype=dtype, device=DEV)
    t = buf[off:off + n].view(store)
    inv = [order.index(i) for i in range(nd)]
    return t.permute(*inv)


def fill_(t, rng, lo=-1.0, hi=1.0, normal=True):
    g = torch.Generator(device=DEV).manual_seed(int(rng.integers(1 << 30)))
    src = torch.empty(t.shape, device=DEV)
    if normal:
        src.normal_(generator=g)
    else:
        src.uniform_(lo, hi, generator=g)
    t.copy_(src.to(t.dtype))
    return t


@pytest.mark.parametrize("seed", range(40))
def test_random_combine(seed):
    rng = np.random.default_rng(1000 + seed)
    dt = TYPES[seed % 3]
    N = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 16, 33]))
    G, B, Hc = int(rng.integers(1, 4)), int(rng.integers(1, 7)), int(rng.integers(1, 10))
    D = int(rng.choice([1, 2, 3, 7, 8, 64, 100, 128, 256, 512, 600]))
    base = str(rng.choice(["e", "2"]))
    sanitize = bool(rng.integers(2))
    ret = bool(rng.integers(2))
    o = fill_(strided((G, N, B, Hc, D), dt, rng), rng)
    lse = fill_(strided((G, N, B, Hc), torch.float32, rng, 0), rng, -10, 25, normal=False)
    if rng.integers(2):  # neutral ranks and a few non-finite values
        lse[0, 0, 0, 0] = -float("inf")
        if N > 1:
            lse[-1, -1, -1, -1] = float(rng.choice([float("nan"), float("inf"), -float("inf")]))
        o[tuple(int(rng.integers(n)) for n in o.shape)] = float(rng.choice([float("nan"), float("inf")]))
    out = strided((G, B, Hc, D), dt, rng)
    out_lse = strided((G, B, Hc), torch.float32, rng, 0) if ret else None
    binding.lse_combine(o, lse, out, out_lse, base=base, sanitize=sanitize)
    want, want_lse = oracle.combine(ORACLE_DT[dt], to_np(o), to_np(lse), base=base, sanitize=sanitize)
    torch.cuda.synchronize()
    if N == 1:
        assert torch.equal(out.contiguous().view(torch.uint8), o[:, 0].contiguous().view(torch.uint8))
    else:
        assert_merge_close(out, want)
    if ret:
        assert_lse_close(out_lse, want_lse)


@pytest.mark.parametrize("seed", range(20))
def test_random_pack(seed):
    rng = np.random.default_rng(2000 + seed)
    dt = TYPES[seed % 3]
    e = torch.empty((), dtype=dt).element_size()
    lpd = 4 // e
    N = int(rng.choice([1, 2, 3, 4, 8]))
    H = N * int(rng.integers(1, 6))
    G, B = int(rng.integers(1, 4)), int(rng.integers(1, 6))
    D = lpd * int(rng.integers(1, 80))
    Hpr = H // N
    o = fill_(strided((G, B, H, D), dt, rng), rng)
    lse = fill_(strided((G, B, H), torch.float32, rng, 0), rng)
    if rng.integers(2):
        # peer-major interleaved with `pad` spare elements per row
        pad = lpd * int(rng.integers(0, 3))
        W = D + lpd + pad
        buf = torch.empty((G, N, B, Hpr, W), dtype=dt, device=DEV)
        buf.view(torch.uint8).fill_(0x6B)
        words = buf.view(torch.float32)
        binding.pack_send(o, lse, buf[..., :D], words[..., D // lpd])
        want = np.empty(buf.shape, dtype=NP_PAYLOAD[dt])
        want.view(np.uint8)[...] = 0x6B
        oracle.pack(ORACLE_DT[dt], N, to_np(o), to_np(lse), want[..., :D], want.view(np.float32)[..., D // lpd])
        torch.cuda.synchronize()
        assert_bytes_equal(buf, want, "interleaved send buffer")
    else:
        po = torch.empty((G, B, Hpr, N, D), dtype=dt, device=DEV)
        po.view(torch.uint8).fill_(0x3C)
        st = torch.full((G, B, Hpr, N, 2), -3.25, device=DEV)
        binding.pack_send(o, lse, po.permute(0, 3, 1, 2, 4), st[..., 0].permute(0, 3, 1, 2))
        want = np.empty(po.shape, dtype=NP_PAYLOAD[dt])
        want.view(np.uint8)[...] = 0x3C
        wst = np.full(st.shape, -3.25, dtype=np.float32)
        oracle.pack(ORACLE_DT[dt], N, to_np(o), to_np(lse), want.transpose(0, 3, 1, 2, 4),
                    wst[..., 0].transpose(0, 3, 1, 2))
        torch.cuda.synchronize()
        assert_bytes_equal(po, want, "peer-inside payload")
        assert_bytes_equal(st, wst, "stats (slot 1 untouched)")


@pytest.mark.parametrize("seed", range(20))
def test_random_unpack_combine(seed):
    rng = np.random.default_rng(3000 + seed)
    dt = TYPES[seed % 3]
    e = torch.empty((), dtype=dt).element_size()
    lpd = 4 // e
    N = int(rng.choice([1, 2, 3, 4, 6, 8, 12]))
    G, B, Hpr = int(rng.integers(1, 4)), int(rng.integers(1, 6)), int(rng.integers(1, 9))
    D = lpd * int(rng.choice([1, 3, 16, 32, 64, 128, 256]))
    pad = lpd * int(rng.integers(0, 3))
    W = D + lpd + pad
    base = str(rng.choice(["e", "2"]))
    sanitize = bool(rng.integers(2))
    recv = torch.empty((G, N, B, Hpr, W), dtype=dt, device=DEV)
    recv.view(torch.uint8).zero_()
    fill_(recv[..., :D], rng)
    words = recv.view(torch.float32)
    fill_(words[..., D // lpd], rng, -5, 20, normal=False)
    if rng.integers(2):
        words[0, 0, 0, 0, D // lpd] = -float("inf")
    out = strided((G, B, Hpr, D), dt, rng)
    out_lse = torch.empty((G, B, Hpr), device=DEV)
    binding.unpack_combine(recv[..., :D + lpd], D, out, out_lse, base=base, sanitize=sanitize)
    r_np = to_np(recv)[..., :D + lpd]
    want, want_lse = oracle.unpack_combine(ORACLE_DT[dt], r_np, D, base=base, sanitize=sanitize)
    torch.cuda.synchronize()
    if N == 1:
        assert torch.equal(out.contiguous().view(torch.uint8),
                           recv[:, 0, ..., :D].contiguous().view(torch.uint8))
    else:
        assert_merge_close(out, want)
    assert_lse_close(out_lse, want_lse)
