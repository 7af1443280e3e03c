"""GPU parity of each rank's decode attention over its round-robin share of the
KV cache (the step that produces the merge's inputs), against the oracle's
split attention, and the whole one-GPU DCP decode (attention per rank, pack,
exchange view, combine) against unsplit attention.

Attention tolerances (fp32 arithmetic over 16-bit inputs, written here): the
payload output as for the merges (tests/parity.py); the LSE within
2e-4 + 1e-5 |lse|: fp32 dot products of up to 256 terms whose magnitudes sum
to ~sm_scale * D (about 1e-4 absolute at worst) plus the rounding of the
log-sum-exp itself.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build, layouts

from parity import assert_merge_close, to_f64, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    binding.load()
    oracle.build()


def local_caches(K, N):
    """Global cache [B, L, Hkv, D] -> every rank's local cache [N, B, ceil(L/N), Hkv, D]
    (token i of rank r is global token i*N + r; the tail is zero padding)."""
    B, L, Hkv, D = K.shape
    lc = (L + N - 1) // N
    out = torch.zeros((N, B, lc, Hkv, D), dtype=K.dtype, device=K.device)
    for r in range(N):
        part = K[:, r::N]
        out[r, :, :part.shape[1]] = part
    return out


def make_case(N, B, H, Hkv, D, lens, dtype, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    L = max(max(lens), 1)
    q = torch.randn((B, H, D), generator=g, device=DEV).to(dtype)
    K = torch.randn((B, L, Hkv, D), generator=g, device=DEV).to(dtype)
    V = torch.randn((B, L, Hkv, D), generator=g, device=DEV).to(dtype)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return q, K, V, seq, L


def run_attention(q, K, V, seq, L, N, scale, base, split):
    B, H, D = q.shape
    Hkv = K.shape[2]
    k, v = local_caches(K, N), local_caches(V, N)
    o = torch.empty((N, B, H, D), dtype=q.dtype, device=DEV)
    lse = torch.empty((N, B, H), dtype=torch.float32, device=DEV)
    nbytes = binding.workspace_bytes(N, B, H, D, L, split)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV) if nbytes else None
    binding.decode_attention(q, k, v, seq, L, o, lse, scale, base=base, split_tokens=split, workspace=ws)
    return o, lse


def oracle_partials(q, K, V, lens, N, scale, base):
    B, H, D = q.shape
    Hkv = K.shape[2]
    gq = H // Hkv
    qn, Kn, Vn = to_f64(q), to_f64(K), to_f64(V)
    want = np.zeros((N, B, H, D))
    want_lse = np.zeros((N, B, H))
    for b in range(B):
        for h in range(H):
            O, l = oracle.split_attention(qn[b, h], Kn[b, :lens[b], h // gq], Vn[b, :lens[b], h // gq], N,
                                          scale, base=base)
            want[:, b, h], want_lse[:, b, h] = O, l
    return want, want_lse


def assert_attn_lse(got, want, what="lse"):
    g = to_f64(got).reshape(want.shape)
    ninf = want == -np.inf
    assert np.array_equal(g == -np.inf, ninf), f"{what}: empty-rank positions differ"
    d = np.abs(g[~ninf] - want[~ninf])
    bad = d > 2e-4 + 1e-5 * np.abs(want[~ninf])
    assert not bad.any(), f"{what}: {int(bad.sum())} values off, max {d.max():.3e}"


CASES = [
    # N, B, H, Hkv, D, lengths, dtype, base, split_tokens
    (4, 3, 4, 4, 128, [0, 1, 3, 4, 5, 200, 1111], torch.bfloat16, "e", 16),
    (4, 3, 4, 4, 128, [0, 1, 3, 4, 5, 200, 1111], torch.bfloat16, "2", 4096),
    (2, 2, 8, 2, 64, [7, 64, 129, 300], torch.float16, "e", 32),
    (8, 2, 4, 1, 256, [3, 9, 17, 500], torch.bfloat16, "2", 40),
    (3, 2, 16, 2, 128, [1, 2, 1000], torch.float16, "2", 100),
    (1, 2, 2, 2, 128, [0, 1, 77], torch.bfloat16, "e", 8),
    # grouped-query heads (the tensor-core path for D <= 128): block tails,
    # splits that are and are not multiples of the 16-token block
    (4, 3, 8, 4, 128, [0, 1, 15, 16, 17, 33, 1500], torch.bfloat16, "e", 48),
    (2, 2, 32, 4, 128, [5, 100, 257, 4097], torch.bfloat16, "2", 1000),
    (4, 2, 16, 4, 64, [1, 31, 64, 999], torch.float16, "e", 24),
    (1, 2, 8, 1, 128, [3, 700], torch.bfloat16, "2", 4096),
    (3, 2, 4, 2, 64, [2, 18, 95], torch.bfloat16, "e", 7),
    (2, 3, 16, 2, 256, [1, 9, 300], torch.float16, "e", 64),
    # 16 query heads per KV head (two blocks of 8 fragment rows)
    (2, 2, 32, 2, 128, [3, 250, 1025], torch.bfloat16, "2", 96),
    (3, 2, 16, 1, 64, [1, 17, 400], torch.float16, "e", 40),
    (3, 1, 8, 4, 256, [77], torch.bfloat16, "2", 16),
]


@pytest.mark.parametrize("N,B,H,Hkv,D,lens,dtype,base,split", CASES)
def test_rank_partials_match_oracle(N, B, H, Hkv, D, lens, dtype, base, split):
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, dtype, seed=N * 100 + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_attention(q, K, V, seq, L, N, scale, base, split)
    want, want_lse = oracle_partials(q, K, V, lens, N, scale, base)
    torch.cuda.synchronize()
    assert_merge_close(o, want, "rank partial O")
    assert_attn_lse(lse, want_lse)


def test_lengths_above_the_bound_are_clamped():
    N, D = 2, 64
    q, K, V, seq, L = make_case(N, 2, 2, 2, D, [10, 30], torch.bfloat16, seed=5)
    seq_big = torch.tensor([10, 10_000], dtype=torch.int32, device=DEV)
    o, lse = run_attention(q, K, V, seq_big, 30, N, 0.125, "e", 8)
    want, want_lse = oracle_partials(q, K, V, [10, 30], N, 0.125, "e")
    torch.cuda.synchronize()
    assert_merge_close(o, want)
    assert_attn_lse(lse, want_lse)


@pytest.mark.parametrize("base", ["e", "2"])
def test_whole_dcp_decode_equals_unsplit_attention(base):
    """Attention per rank -> peer-inside pack -> exchange view -> combine, all on
    one GPU, equals single-query softmax attention over the whole sequence."""
    N, H, Hkv, D = 4, 16, 4, 128
    lens = [1, 3, 57, 640, 2049, 4]
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, torch.bfloat16, seed=77)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_attention(q, K, V, seq, L, N, scale, base, 256)       # [N,B,H,D], [N,B,H]
    H_pr = H // N
    partial_o, stats = layouts.alloc_peer_inside(N, B, H_pr, N, D, torch.bfloat16, DEV)
    binding.pack_send(o, lse, *layouts.peer_inside_send_views(partial_o, stats))
    ro, rl = layouts.exchange_peer_inside(partial_o, stats)
    out = torch.empty((N, B, H_pr, D), dtype=torch.bfloat16, device=DEV)
    out_lse = torch.empty((N, B, H_pr), dtype=torch.float32, device=DEV)
    binding.lse_combine(ro, rl, out, out_lse, base=base)
    torch.cuda.synchronize()
    # destination d holds heads [d*H_pr, (d+1)*H_pr)
    got = out.permute(1, 0, 2, 3).reshape(B, H, D)
    got_lse = out_lse.permute(1, 0, 2).reshape(B, H)
    qn, Kn, Vn = to_f64(q), to_f64(K), to_f64(V)
    want = np.zeros((B, H, D))
    want_lse = np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            s = (Kn[b, :lens[b], h // (H // Hkv)] @ qn[b, h]) * scale
            m = s.max()
            p = np.exp(s - m)
            want[b, h] = (p / p.sum()) @ Vn[b, :lens[b], h // (H // Hkv)]
            want_lse[b, h] = (m + math.log(p.sum())) / (math.log(2.0) if base == "2" else 1.0)
    # the merge itself, exactly as the oracle merges the GPU's own bf16 partials
    po_np = to_np(partial_o)
    st_np = stats.cpu().numpy()
    m_want, m_want_lse = oracle.combine("bf16", po_np.transpose(3, 0, 1, 2, 4), st_np[..., 0].transpose(3, 0, 1, 2),
                                        base=base)
    assert_merge_close(out, m_want, "merge of the GPU partials")
    # against unsplit attention: the pipeline rounds twice (each rank's partial
    # to bf16, then the merged row), so per element |d| <= 2^-8 (|want| +
    # sum_r w_r |O_r|) + 1e-5, with w_r and O_r the oracle's per-rank values
    parts, plse = oracle_partials(q, K, V, lens, N, scale, "e")
    with np.errstate(invalid="ignore"):
        gl = np.logaddexp.reduce(plse, axis=0)
        w = np.nan_to_num(np.exp(plse - gl[None]), nan=0.0)
    spread = (w[..., None] * np.abs(parts)).sum(axis=0)
    d = np.abs(to_f64(got) - want)
    bound = 2.0 ** -8 * (np.abs(want) + spread) + 1e-5
    assert (d <= bound).all(), f"merged attention: worst excess {(d - bound).max():.3e}"
    assert d.max() / np.abs(want).max() <= 2e-2
    assert_attn_lse(got_lse, want_lse, "merged lse")


@pytest.mark.parametrize("name,split", [("mha_decode_attention", 1024), ("gqa_decode_attention", 2048)])
def test_decode_attention_workload_full_size_sampled(name, split):
    """The benchmark's workloads (N=4, B=64, H=32 over 32 or 4 KV heads, D=128,
    lengths up to 16384) in their launch configuration (splits of 1024 / 2048
    local tokens): sampled (request, head) rows of every rank against the oracle."""
    from decode_context_attention_gb300.workloads import generate_attention

    a = generate_attention(name, device=DEV)
    c = a["cfg"]
    N, B, H, Hkv, D = c["N"], c["B"], c["H"], c["Hkv"], c["D"]
    scale = 1.0 / math.sqrt(D)
    o = torch.empty((N, B, H, D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((N, B, H), dtype=torch.float32, device=DEV)
    nbytes = binding.workspace_bytes(N, B, H, D, a["max_len"], split)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    binding.decode_attention(a["q"], a["k"], a["v"], a["seq_lens"], a["max_len"], o, lse, scale,
                             base=c["base"], split_tokens=split, workspace=ws)
    torch.cuda.synchronize()
    lens = a["seq_lens"].cpu().tolist()
    rng = np.random.default_rng(3)
    picks = [(int(b), int(h)) for b, h in zip(rng.integers(0, B, 24), rng.integers(0, H, 24))]
    picks += [(int(np.argmax(lens)), 0), (int(np.argmin(lens)), H - 1)]
    for b, h in picks:
        L = lens[b]
        hk = h // (H // Hkv)
        # rebuild the global sequence: global token t = local token t // N of rank t % N
        kg = torch.stack([a["k"][t % N, b, t // N, hk] for t in range(L)]) if L < 64 else None
        if kg is None:
            idx = torch.arange(L, device=DEV)
            kg = a["k"][idx % N, b, idx // N, hk]
            vg = a["v"][idx % N, b, idx // N, hk]
        else:
            vg = torch.stack([a["v"][t % N, b, t // N, hk] for t in range(L)])
        O, l = oracle.split_attention(to_f64(a["q"][b, h]), to_f64(kg), to_f64(vg), N, scale, base=c["base"])
        assert_merge_close(o[:, b, h], O, f"row b={b} h={h}")
        assert_attn_lse(lse[:, b, h], l, f"lse b={b} h={h}")


def paged_caches(k, v, page_size, seed, spare=3):
    """Scatter local caches [N, B, Lc, Hkv, D] into per-rank page pools
    [N, num_pages, page_size, Hkv, D] with each rank's pages in a shuffled
    order; pages nobody owns hold NaN, so a read of a wrong page shows.
    Returns (k_pages, v_pages, block_table [N, B, max_pages] int32)."""
    N, B, Lc, Hkv, D = k.shape
    max_pages = (Lc + page_size - 1) // page_size
    num_pages = B * max_pages + spare
    g = torch.Generator().manual_seed(seed)
    bt = torch.stack([torch.randperm(num_pages, generator=g)[:B * max_pages] for _ in range(N)])
    pools = []
    for src in (k, v):
        pad = torch.zeros((N, B, max_pages * page_size, Hkv, D), dtype=src.dtype, device=DEV)
        pad[:, :, :Lc] = src
        pool = torch.full((N, num_pages, page_size, Hkv, D), float("nan"), device=DEV).to(src.dtype)
        for r in range(N):
            pool[r, bt[r].to(DEV)] = pad[r].reshape(B * max_pages, page_size, Hkv, D)
        pools.append(pool)
    return pools[0], pools[1], bt.view(N, B, max_pages).to(torch.int32).to(DEV)


PAGED = [
    # N, H, Hkv, D, lengths, dtype, base, split_tokens, page_size
    (4, 8, 1, 128, [0, 5, 700], torch.bfloat16, "e", 64, 16),
    (2, 4, 4, 64, [33, 130], torch.float16, "2", 1000, 1),
    (3, 16, 2, 256, [9, 300], torch.bfloat16, "e", 40, 64),
    (2, 8, 4, 256, [77, 5], torch.float16, "2", 16, 8),
    (2, 32, 2, 128, [1, 513], torch.bfloat16, "2", 128, 32),
]


@pytest.mark.parametrize("N,H,Hkv,D,lens,dtype,base,split,page_size", PAGED)
def test_paged_caches_give_the_contiguous_result(N, H, Hkv, D, lens, dtype, base, split, page_size):
    """The same partials from paged caches as from contiguous ones, bit for bit
    (the kernels differ only in where a token's row is read), and the oracle's."""
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, dtype, seed=31 * N + D + page_size)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_attention(q, K, V, seq, L, N, scale, base, split)
    kp, vp, bt = paged_caches(local_caches(K, N), local_caches(V, N), page_size, seed=page_size)
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)
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


STRIDED = [
    # N, H, Hkv, D, lengths, dtype, split_tokens, cache layout, paged page size (0: contiguous)
    (3, 4, 4, 128, [0, 9, 300], torch.bfloat16, 64, "kv_interleaved", 0),      # CUDA cores
    (2, 16, 2, 128, [5, 700], torch.float16, 128, "head_major", 0),            # tensor cores
    (2, 4, 2, 256, [33, 90], torch.bfloat16, 32, "kv_interleaved", 0),         # two heads at D = 256
    (4, 8, 2, 64, [1, 250, 513], torch.bfloat16, 4096, "head_major", 0),       # one split
    (2, 8, 2, 128, [17, 400], torch.bfloat16, 48, "kv_interleaved", 16),       # paged, interleaved pool
]


@pytest.mark.parametrize("N,H,Hkv,D,lens,dtype,split,layout,page", STRIDED)
def test_strided_operands_give_the_contiguous_result(N, H, Hkv, D, lens, dtype, split, layout, page):
    """Operands as serving engines hold them: q sliced out of a fused
    [B, H + 2 Hkv, D] projection, K and V interleaved in one cache
    ([.., 2, Hkv, D] per token) or head-major ([.., Hkv, Lc, D]), the output
    rows padded and the LSE a strided slot of a [.., 2] stats array.  The
    kernels only follow the strides, so the results equal the contiguous
    call's bit for bit."""
    B = len(lens)
    q, K, V, seq, L = make_case(N, B, H, Hkv, D, lens, dtype, seed=500 + D + H)
    scale = 1.0 / math.sqrt(D)
    base = "2" if page else "e"
    o_ref, lse_ref = run_attention(q, K, V, seq, L, N, scale, base, split)

    fused = torch.randn((B, H + 2 * Hkv, D), device=DEV).to(dtype)
    fused[:, :H] = q
    qs = fused[:, :H]
    k_loc, v_loc = local_caches(K, N), local_caches(V, N)           # [N, B, Lc, Hkv, D]
    if page:
        k_loc, v_loc, bt = paged_caches(k_loc, v_loc, page, seed=page)  # pools [N, P, page, Hkv, D]
    if layout == "kv_interleaved":
        kv = torch.empty(k_loc.shape[:3] + (2,) + k_loc.shape[3:], dtype=dtype, device=DEV)
        kv[:, :, :, 0], kv[:, :, :, 1] = k_loc, v_loc
        ks, vs = kv[:, :, :, 0], kv[:, :, :, 1]
    else:
        ks = k_loc.permute(0, 1, 3, 2, 4).contiguous().permute(0, 1, 3, 2, 4)
        vs = v_loc.permute(0, 1, 3, 2, 4).contiguous().permute(0, 1, 3, 2, 4)
    assert not ks.is_contiguous() and not qs.is_contiguous()
    obuf = torch.full((N, B, H, D + 24), 7.0, device=DEV).to(dtype)
    lbuf = torch.full((N, B, H, 2), 7.0, device=DEV)
    o, lse = obuf[..., :D], lbuf[..., 0]
    nbytes = binding.workspace_bytes(N, B, H, D, L, split)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV) if nbytes else None
    if page:
        binding.decode_attention_paged(qs, ks, vs, bt, seq, L, o, lse, scale, base=base, split_tokens=split,
                                       workspace=ws)
    else:
        binding.decode_attention(qs, ks, vs, seq, L, o, lse, scale, base=base, split_tokens=split, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o.contiguous().view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.contiguous().view(torch.int32), lse_ref.view(torch.int32))
    # nothing outside the views was written
    assert bool((obuf[..., D:] == 7.0).all()) and bool((lbuf[..., 1] == 7.0).all())
