"""Seeded random sweep of the per-rank decode attention: random rank counts,
batch, query heads per KV head (1..16), head dims, lengths (including 0 and
lengths off every block grid), split sizes, bases, 16-bit types and contiguous
or paged caches (random page sizes, shuffled pools), against the oracle's
split attention (tolerances of tests/test_attention_gpu.py)."""
import math

import numpy as np
import pytest
import torch

from decode_context_attention_gb300 import binding, build

from parity import assert_merge_close
from test_attention_gpu import (assert_attn_lse, local_caches, make_case, oracle_partials, paged_caches,
                                run_attention)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()


@pytest.mark.parametrize("seed", range(24))
def test_random_attention(seed):
    rng = np.random.default_rng(7000 + seed)
    gq = int(rng.choice([1, 2, 4, 8, 16]))
    D = int(rng.choice([64, 128] if gq == 16 else [64, 128, 256]))
    Hkv = int(rng.choice([1, 2, 3]))
    H = gq * Hkv
    N = int(rng.choice([1, 2, 3, 4, 8]))
    B = int(rng.integers(1, 4))
    lens = [int(x) for x in rng.choice([0, 1, 7, 16, 17, 63, 100, 257, 900, 1500], size=B)]
    dtype = [torch.bfloat16, torch.float16][seed % 2]
    base = str(rng.choice(["e", "2"]))
    split = int(rng.choice([5, 16, 33, 128, 4096]))
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, dtype, seed=9000 + seed)
    scale = 1.0 / math.sqrt(D)
    if rng.integers(2):
        o, lse = run_attention(q, K, V, seq, L, N, scale, base, split)
    else:
        page = int(rng.choice([1, 4, 16, 64]))
        kp, vp, bt = paged_caches(local_caches(K, N), local_caches(V, N), page, seed=seed)
        o = torch.empty((N, B, H, D), dtype=dtype, device=DEV)
        lse = torch.empty((N, B, H), device=DEV)
        nbytes = binding.workspace_bytes(N, B, H, D, L, split)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV) if nbytes else None
        binding.decode_attention_paged(q, kp, vp, bt, seq, L, o, lse, scale, base=base, split_tokens=split,
                                       workspace=ws)
    want, want_lse = oracle_partials(q, K, V, lens, N, scale, base)
    torch.cuda.synchronize()
    assert_merge_close(o, want, f"seed {seed} (N={N} H={H} Hkv={Hkv} D={D} lens={lens} split={split})")
    assert_attn_lse(lse, want_lse)
