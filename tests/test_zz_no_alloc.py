"""The attention entry point for callers that cannot allocate device memory.

Some callers of this library may not allocate at the point where they run
the attention (a memory pool sized up front, a serving loop that forbids
allocation, a host runtime without an allocator), so they cannot hand in a
workspace.  dcp_decode_attention_noalloc keeps the split partials in scratch
built into the library instead.  Called through the C ABI, its output must
equal the workspace entry point's on two calls in a row (the second on other
data, so nothing of the first call leaks into it), and sizes that need more
than the built-in scratch must be refused with a clear message.

This file is collected last, so a run that stops at the first failure has
already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from decode_context_attention_gb300 import binding, build

from parity import assert_merge_close, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def case(seed, lens, N=4, H=8, Hkv=4, D=128):
    g = torch.Generator(device=DEV).manual_seed(seed)
    B = len(lens)
    L = max(lens)
    lc = (L + N - 1) // N
    q = torch.randn((B, H, D), generator=g, device=DEV).to(torch.bfloat16)
    k = torch.randn((N, B, lc, Hkv, D), generator=g, device=DEV).to(torch.bfloat16)
    v = torch.randn((N, B, lc, Hkv, D), generator=g, device=DEV).to(torch.bfloat16)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return q, k, v, seq, L


def raw_args(q, k, v, seq, L, o, lse, scale, split, base):
    B, H, D = q.shape
    N, _, _, Hkv, _ = k.shape
    return (2, N, B, H, Hkv, D,
            q.data_ptr(), q.stride(0), q.stride(1),
            k.data_ptr(), k.stride(0), k.stride(1), k.stride(2), k.stride(3),
            v.data_ptr(), v.stride(0), v.stride(1), v.stride(2), v.stride(3),
            seq.data_ptr(), L, scale, split,
            o.data_ptr(), o.stride(0), o.stride(1), o.stride(2),
            lse.data_ptr(), lse.stride(0), lse.stride(1), lse.stride(2), base)


def test_no_alloc_entry_point_matches_the_workspace_entry_point():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    lib = binding.load()
    stream = torch.cuda.current_stream().cuda_stream
    split = 32  # several splits per rank, so the scratch is used
    for call, (seed, lens) in enumerate([(101, [5, 700, 129, 64]), (202, [1000, 3, 400])]):
        q, k, v, seq, L = case(seed, lens)
        N, B, H, D = k.shape[0], q.shape[0], q.shape[1], q.shape[2]
        scale = 1.0 / math.sqrt(D)
        base = call  # base e on the first call, base 2 on the second
        need = binding.workspace_bytes(N, B, H, D, L, split)
        assert need > 0
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        o_ref = torch.empty((N, B, H, D), dtype=torch.bfloat16, device=DEV)
        lse_ref = torch.empty((N, B, H), dtype=torch.float32, device=DEV)
        binding.decode_attention(q, k, v, seq, L, o_ref, lse_ref, scale, base="2" if base else "e",
                                 split_tokens=split, workspace=ws)
        o = torch.full((N, B, H, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((N, B, H), float("nan"), dtype=torch.float32, device=DEV)
        st = lib.dcp_decode_attention_noalloc(*raw_args(q, k, v, seq, L, o, lse, scale, split, base), stream)
        assert st == 0, binding.dcp_last_error_message()
        torch.cuda.synchronize()
        # the same kernels on the same inputs: within the merge tolerance (in
        # fact bit for bit)
        assert_merge_close(o, to_f64(o_ref), f"call {call + 1} O")
        got_l, want_l = to_f64(lse), to_f64(lse_ref)
        assert np.array_equal(got_l == -np.inf, want_l == -np.inf)
        fin = np.isfinite(want_l)
        assert np.abs(got_l[fin] - want_l[fin]).max(initial=0.0) <= 1e-5
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))


def test_no_alloc_entry_point_refuses_sizes_beyond_its_scratch():
    build.build()
    lib = binding.load()
    q, k, v, seq, L = case(7, [64, 64])
    o = torch.empty((4, 2, 8, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((4, 2, 8), dtype=torch.float32, device=DEV)
    # a bound of 2^21 tokens in splits of 8 needs about 1 GiB of scratch
    args = list(raw_args(q, k, v, seq, 1 << 21, o, lse, 0.1, 8, 0))
    st = lib.dcp_decode_attention_noalloc(*args, torch.cuda.current_stream().cuda_stream)
    assert st == 1  # DCP_ERR_INVALID_ARG
    assert "scratch" in binding.dcp_last_error_message()


# A process of its own: it resets the device, which would pull the memory out
# from under every tensor of the test session.  Only the CUDA runtime (through
# ctypes) and the library run in it.
_RESET_SCRIPT = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from decode_context_attention_gb300 import binding

lib = binding.load()
cudart_path = next(line.split()[-1] for line in open("/proc/self/maps") if "libcudart.so" in line)
rt = ctypes.CDLL(cudart_path)
rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
rt.cudaFree.argtypes = [ctypes.c_void_p]

def ok(e, what):
    if e != 0:
        raise SystemExit(f"{what} failed with CUDA error {e}")

N, B, H, Hkv, D, split = 4, 3, 8, 4, 128, 32
lens = np.array([700, 5, 129], dtype=np.int32)
L = int(lens.max())
lc = (L + N - 1) // N
rng = np.random.default_rng(5)
def bf16(shape):
    f = rng.standard_normal(shape).astype(np.float32)
    return ((f.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
host = {"q": bf16((B, H, D)), "k": bf16((N, B, lc, Hkv, D)), "v": bf16((N, B, lc, Hkv, D)), "seq": lens}
need = binding.workspace_bytes(N, B, H, D, L, split)
assert need > 0

def run(noalloc):
    dev = {}
    for name, a in host.items():
        p = ctypes.c_void_p()
        ok(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
        ok(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, 1), "cudaMemcpy H2D")
        dev[name] = p.value
    sizes = {"o": N * B * H * D * 2, "lse": N * B * H * 4, "ws": need}
    for name, n in sizes.items():
        p = ctypes.c_void_p()
        ok(rt.cudaMalloc(ctypes.byref(p), n), "cudaMalloc")
        dev[name] = p.value
    args = (2, N, B, H, Hkv, D, dev["q"], H * D, D,
            dev["k"], B * lc * Hkv * D, lc * Hkv * D, Hkv * D, D,
            dev["v"], B * lc * Hkv * D, lc * Hkv * D, Hkv * D, D,
            dev["seq"], L, 1.0 / D ** 0.5, split,
            dev["o"], B * H * D, H * D, D, dev["lse"], B * H, H, 1, 1)
    if noalloc:
        st = lib.dcp_decode_attention_noalloc(*args, None)
    else:
        st = lib.dcp_decode_attention(*args, dev["ws"], need, None)
    assert st == 0, binding.dcp_last_error_message()
    ok(rt.cudaDeviceSynchronize(), "kernels")
    o = np.empty(N * B * H * D, dtype=np.uint16)
    lse = np.empty(N * B * H, dtype=np.uint32)
    ok(rt.cudaMemcpy(o.ctypes.data, dev["o"], o.nbytes, 2), "cudaMemcpy D2H")
    ok(rt.cudaMemcpy(lse.ctypes.data, dev["lse"], lse.nbytes, 2), "cudaMemcpy D2H")
    for p in dev.values():
        ok(rt.cudaFree(ctypes.c_void_p(p)), "cudaFree")
    return o, lse

ok(rt.cudaSetDevice(0), "cudaSetDevice")
for attempt in range(2):
    want_o, want_l = run(noalloc=False)
    got_o, got_l = run(noalloc=True)
    assert np.array_equal(want_o, got_o) and np.array_equal(want_l, got_l), f"attempt {attempt}: differs"
    assert (want_l != 0).any()
    if attempt == 0:
        ok(rt.cudaDeviceReset(), "cudaDeviceReset")
print("noalloc ok across a device reset")
'''


def test_no_alloc_entry_point_after_a_device_reset():
    # cudaDeviceReset ends the context the scratch array's address was looked
    # up in; the next call must find the array of the new context, and give
    # the workspace entry point's result bit for bit again
    import os
    import subprocess
    import sys

    build.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _RESET_SCRIPT, root], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "noalloc ok across a device reset" in r.stdout
