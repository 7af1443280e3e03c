"""Several host threads driving the library at once, each on its own CUDA
stream: the interleaved pack + fused unpack+combine of eight different
payload types, rank counts and head dims (so eight different kernel choices,
and the per-device launch-shape caches are filled from several threads),
repeated, must give the bytes the same steps give one after another on the
default stream."""
import threading

import pytest
import torch

from decode_context_attention_gb300 import binding, build, layouts

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8 = torch.float8_e4m3fn
CASES = [(torch.float32, 2, 128), (torch.float16, 3, 40), (torch.bfloat16, 8, 512), (FP8, 4, 256),
         (torch.float32, 33, 64), (torch.bfloat16, 5, 1000), (torch.float16, 8, 514), (FP8, 16, 12)]


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()


def make(case, seed):
    dtype, N, D = case
    g = torch.Generator(device=DEV).manual_seed(seed)
    B, H = 16, 4 * N
    o = torch.randn((N, B, H, D), generator=g, device=DEV).clamp(-440, 440).to(dtype)
    lse = torch.empty((N, B, H), device=DEV).uniform_(-10, 10, generator=g)
    lse[0, 3, :] = -float("inf")
    return o, lse


def step(o, lse, stream):
    """Pack all N source ranks into peer-major interleaved rows, then merge
    every destination's receive rows; allocations follow the current stream."""
    N, B, H, D = o.shape
    lpd = binding.dcp_lse_pack_dim(binding.DTYPE_CODES[o.dtype])
    send = torch.empty((N, N, B, H // N, D + lpd), dtype=o.dtype, device=DEV)
    out = torch.empty((N, B, H // N, D), dtype=o.dtype, device=DEV)
    out_lse = torch.empty((N, B, H // N), device=DEV)
    binding.pack_send(o, lse, *layouts.peer_major_views(send, D), stream=stream)
    binding.unpack_combine(layouts.exchange_peer_major(send), D, out, out_lse, base="2", stream=stream)
    return send, out, out_lse


def as_bytes(t):
    return t.contiguous().view(torch.uint8).cpu()


def test_concurrent_threads_on_their_own_streams_match_sequential_calls():
    inputs = [make(c, 300 + i) for i, c in enumerate(CASES)]
    want = [[as_bytes(t) for t in step(o, lse, None)] for o, lse in inputs]
    torch.cuda.synchronize()
    got, errors = [None] * len(CASES), []
    barrier = threading.Barrier(len(CASES))

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                o, lse = inputs[i]
                barrier.wait()
                for _ in range(8):
                    res = step(o, lse, s)
                s.synchronize()
                got[i] = [as_bytes(t) for t in res]
        except BaseException as e:  # reported by the main thread
            errors.append((i, e))
            barrier.abort()

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, case in enumerate(CASES):
        for name, a, b in zip(("send", "out", "out_lse"), got[i], want[i]):
            assert torch.equal(a, b), f"{case}: {name} differs from the sequential result"
