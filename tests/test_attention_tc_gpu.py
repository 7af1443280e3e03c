"""GPU parity of the grouped-query decode attention's tensor-core path
(tcgen05, D = 128, 2 to 16 query heads per KV head, split_tokens a multiple
of 128) against the oracle's split attention: tile edges, one and several
splits, both payload types and LSE bases, paged caches of every page size
the path takes (bit-identical to the contiguous call), page indices outside
the pool, stale cache rows past each rank's length, scores that keep moving
the reference max, and a bounded wait that runs out.  Tolerances as in test_attention_gpu.py.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build

from parity import assert_merge_close, to_f64
from test_attention_gpu import (assert_attn_lse, local_caches, make_case, oracle_partials, paged_caches,
                                run_attention)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


TC_CASES = [
    # N, H, Hkv, D, lengths, dtype, base, split_tokens
    # tile edges around 128 local tokens, several splits of one tile
    (1, 8, 4, 128, [1, 127, 128, 129, 255, 256, 257], torch.bfloat16, "e", 128),
    # every group size, ragged lengths, several splits
    (2, 4, 2, 128, [0, 1, 128, 383, 2000], torch.float16, "e", 256),
    (3, 16, 4, 128, [0, 700, 5000], torch.bfloat16, "2", 128),
    (4, 32, 4, 128, [1, 127, 129, 3000, 4], torch.bfloat16, "e", 512),
    (2, 32, 2, 128, [3, 256, 2049], torch.float16, "2", 128),
    # one split per rank (outputs written directly), lengths past a tile
    (2, 16, 1, 128, [5, 300, 1000], torch.bfloat16, "2", 4096),
    (8, 64, 8, 128, [1, 9, 2500], torch.float16, "e", 1024),
]


@pytest.mark.parametrize("N,H,Hkv,D,lens,dtype,base,split", TC_CASES)
def test_tensor_core_partials_match_oracle(N, H, Hkv, D, lens, dtype, base, split):
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, dtype, seed=900 + N * 10 + H)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_attention(q, K, V, seq, L, N, scale, base, split)
    want, want_lse = oracle_partials(q, K, V, lens, N, scale, base)
    torch.cuda.synchronize()
    assert_merge_close(o, want, "rank partial O")
    assert_attn_lse(lse, want_lse)


PAGED_TC = [
    # N, H, Hkv, lengths, dtype, base, split_tokens, page_size
    (2, 8, 1, [0, 5, 700], torch.bfloat16, "e", 128, 8),
    (3, 16, 2, [9, 300, 1500], torch.float16, "2", 256, 16),
    (4, 32, 4, [1, 129, 2100], torch.bfloat16, "2", 2048, 64),
    (2, 4, 2, [2, 600], torch.bfloat16, "e", 128, 128),
    (2, 16, 1, [77, 1300], torch.float16, "e", 512, 1024),
]


@pytest.mark.parametrize("N,H,Hkv,lens,dtype,base,split,page_size", PAGED_TC)
def test_tensor_core_paged_equals_contiguous(N, H, Hkv, lens, dtype, base, split, page_size):
    """Paged pools (pages shuffled per rank, unowned pages NaN) give the
    contiguous call's partials bit for bit on the tensor-core path, and the
    oracle's."""
    D, B = 128, len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, dtype, seed=40 * N + page_size)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_attention(q, K, V, seq, L, N, scale, base, split)
    kp, vp, bt = paged_caches(local_caches(K, N), local_caches(V, N), page_size, seed=page_size + 1)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    nbytes = binding.workspace_bytes(N, B, H, D, L, split)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV) if nbytes else None
    binding.decode_attention_paged(q, kp, vp, bt, seq, L, o2, lse2, scale, base=base, split_tokens=split,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16))
    assert torch.equal(lse2.view(torch.int32), lse.view(torch.int32))
    want, want_lse = oracle_partials(q, K, V, lens, N, scale, base)
    assert_merge_close(o2, want, "paged rank partial O")
    assert_attn_lse(lse2, want_lse)


def test_tensor_core_page_indices_outside_the_pool_read_zero_rows():
    """A page-table entry outside [0, num_pages) for tokens a rank holds makes
    those tokens' K and V rows read as zeros (score 0, value 0), never memory
    outside the pool."""
    N, H, Hkv, D, page = 2, 8, 2, 128, 16
    lens = [300, 90]
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, torch.bfloat16, seed=11)
    kl, vl = local_caches(K, N), local_caches(V, N)
    kp, vp, bt = paged_caches(kl, vl, page, seed=5)
    num_pages = kp.shape[1]
    bad = [(0, 0, 2), (1, 0, 5), (1, 1, 0)]  # (rank, request, page slot of the table)
    for r, b, j in bad:
        bt[r, b, j] = num_pages + 7 if (r + j) % 2 else -3
    o = torch.empty((N, B, H, D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((N, B, H), dtype=torch.float32, device=DEV)
    split = 128
    nbytes = binding.workspace_bytes(N, B, H, D, L, split)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    binding.decode_attention_paged(q, kp, vp, bt, seq, L, o, lse, 1 / math.sqrt(D), base="e", split_tokens=split,
                                   workspace=ws)
    torch.cuda.synchronize()
    # the oracle over the same caches with those pages' rows zeroed
    K2, V2 = K.clone(), V.clone()
    for r, b, j in bad:
        for i in range(j * page, (j + 1) * page):
            t = i * N + r
            if t < lens[b]:
                K2[b, t] = 0
                V2[b, t] = 0
    want, want_lse = oracle_partials(q, K2, V2, lens, N, 1 / math.sqrt(D), "e")
    assert_merge_close(o, want, "partials with out-of-pool pages")
    assert_attn_lse(lse, want_lse)


def test_tensor_core_ignores_stale_rows_past_each_length():
    """Cache rows past a rank's local length (the rest of the last tile, and
    the next split's rows) may hold anything, NaN and inf included: the
    result equals the one over zero-padded caches bit for bit."""
    N, H, Hkv, D = 3, 16, 2, 128
    lens = [1, 130, 200, 1000]
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, torch.float16, seed=21)
    split = 128
    o_ref, lse_ref = run_attention(q, K, V, seq, L, N, 0.088, "2", split)
    k, v = local_caches(K, N), local_caches(V, N)
    for b, Lb in enumerate(lens):
        for r in range(N):
            ll = Lb // N + (1 if r < Lb % N else 0)
            k[r, b, ll:] = float("nan")
            v[r, b, ll:] = float("inf") if (r + b) % 2 else float("nan")
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    nbytes = binding.workspace_bytes(N, B, H, D, L, split)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    binding.decode_attention(q, k, v, seq, L, o, lse, 0.088, base="2", split_tokens=split, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_tensor_core_rising_scores_move_the_reference_max():
    """Keys that grow along the sequence make the lazily moved reference max
    move (by more than 2^8) within a split, so the transposed output is
    rescaled in place several times; the partials still match the oracle."""
    N, H, Hkv, D = 2, 16, 2, 128
    lens = [4000, 2500, 700, 1]
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, torch.bfloat16, seed=57)
    t = torch.arange(K.shape[1], device=DEV, dtype=torch.float32)
    K = (K.float() * (1.0 + t / 250.0)[None, :, None, None]).to(K.dtype)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_attention(q, K, V, seq, L, N, scale, "2", 1024)
    want, want_lse = oracle_partials(q, K, V, lens, N, scale, "2")
    torch.cuda.synchronize()
    assert_merge_close(o, want, "rank partial O, rising scores")
    assert_attn_lse(lse, want_lse)


_STALL_SCRIPT = r'''
import os, sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, os.path.join(sys.argv[1], "tests"))
import math
import numpy as np
import torch
import oracle
from decode_context_attention_gb300 import binding

binding.load()
dev = "cuda"
g = torch.Generator(device=dev).manual_seed(6)
N, B, H, Hkv, D, L = 2, 1, 8, 2, 128, 300
q = torch.randn((B, H, D), generator=g, device=dev).to(torch.bfloat16)
k = torch.randn((N, B, (L + N - 1) // N, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
v = torch.randn((N, B, (L + N - 1) // N, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
seq = torch.tensor([L], dtype=torch.int32, device=dev)
o = torch.empty((N, B, H, D), dtype=torch.bfloat16, device=dev)
lse = torch.empty((N, B, H), dtype=torch.float32, device=dev)
scale = 1 / math.sqrt(D)
os.environ["DCP_TEST_STALL_LOADS"] = "1"
# 0: a split that is not a multiple of 128 tokens takes the register-tiled
# kernel, which the switch does not touch: no status
binding.decode_attention(q, k, v, seq, L, o, lse, scale, base="e", split_tokens=100,
                         workspace=torch.empty(binding.workspace_bytes(N, B, H, D, L, 100), dtype=torch.uint8,
                                               device=dev))
torch.cuda.synchronize()
assert binding.device_status() == 0
# 1: the tcgen05 kernel (splits of whole 128-token tiles) with every K/V load
# held back: its first wait on them runs out
binding.decode_attention(q, k, v, seq, L, o, lse, scale, base="e", split_tokens=4096)
torch.cuda.synchronize()
st = binding.device_status()
assert st == 7, f"expected DCP_ERR_TIMEOUT, got {st}"
assert binding.device_status() == 0, "the status must clear once read"
# 2: the context is still usable and the next call is right
del os.environ["DCP_TEST_STALL_LOADS"]
binding.decode_attention(q, k, v, seq, L, o, lse, scale, base="e", split_tokens=4096)
torch.cuda.synchronize()
assert binding.device_status() == 0
idx = torch.arange(L, device=dev)
kr = k[idx % N, 0, idx // N, 1].double().cpu().numpy()
vr = v[idx % N, 0, idx // N, 1].double().cpu().numpy()
want, want_lse = oracle.split_attention(q[0, 5].double().cpu().numpy(), kr, vr, N, scale, base="e")
got = o[:, 0, 5].double().cpu().numpy()
assert np.abs(got - want).max() <= 0.02 * np.abs(want).max(), np.abs(got - want).max()
assert np.abs(lse[:, 0, 5].double().cpu().numpy() - want_lse).max() <= 1e-3
print("timeout reported, context usable")
'''


def test_tensor_core_wait_that_runs_out_reports_a_timeout_and_leaves_the_context_usable():
    # held-back loads make the kernel's first bounded wait run out (after 1 s):
    # it must end with DCP_ERR_TIMEOUT in the device status word, not hang or
    # fault.  That the status comes from this call and not from one with a
    # split of 100 tokens also shows which calls take the tcgen05 kernel.
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.pop("DCP_TEST_STALL_LOADS", None)
    r = subprocess.run([sys.executable, "-c", _STALL_SCRIPT, root], capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "timeout reported, context usable" in r.stdout
