"""Absorbed-MLA decode attention on the tensor cores against the fp64 oracle.

Every rank's partial (O_r, lse_r) from dcp_decode_attention_mla is compared,
element by element, with oracle.split_attention_mla on the same seeded
inputs: small cases on every row (ragged tails, ranks owning nothing, one
split and many, both LSE bases, bf16 and fp16, fewer than 128 heads, strided
operands), seeded random shapes on sampled rows, the full-size workload on
sampled rows, a request's rows under both work orders of the persistent
kernel, and the whole one-GPU DCP
decode of the MLA merge's shape (attention -> peer-inside pack -> combine)
against unsplit attention.

Tolerance, from the arithmetic (not fitted): the kernel rounds every
probability once to the payload type before the value product (relative
error <= u, u = 2^-9 for bf16, 2^-12 for fp16), normalises by the fp32 sum
of the unrounded probabilities, and rounds the output once (<= u relative).
So |O - O*|_d <= u sum_t w_t |v_td| + u |O*_d| + the effect of score errors.
The scores are fp32 sums of 576 products, and each of the two CTAs' partial
scores (latent columns [256c, 256c + 256) plus rope columns [512 + 32c,
544 + 32c)) crosses to the other CTA rounded to fp16 in log2 units, both
CTAs rounding alike (relative error <= 2^-11, absolute <= 2^-25 below the
normal range): |ds_t| <= (576 * 2^-24 * sum_i |q_i kv_ti| + 2^-11 (|S_0t| +
|S_1t|)) * sm_scale + 2^-24 ln 2, maximised over t =: E (natural-log units),
which moves lse by at most E and every weight by a factor within
exp(+-2E).  The bounds below take twice each term.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_context_attention_gb300 import binding, build, layouts
from decode_context_attention_gb300.workloads import generate_mla_attention

pytestmark = pytest.mark.gpu
DEV = "cuda"
DK, DV = 576, 512
U = {torch.bfloat16: 2.0 ** -9, torch.float16: 2.0 ** -12}


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    return binding.load()


def global_rows(kv, b, L, N):
    """The request's latent rows in global token order: token t = rank t % N, slot t // N."""
    idx = torch.arange(L, device=kv.device)
    return kv[idx % N, b, idx // N].double().cpu().numpy()


def check_row(got_o, got_lse, q, rows_global, r, N, scale, base, u, what, want=None):
    """One (rank, request, head): the kernel's (O, lse) against the oracle
    (`want` = the oracle's (O [N, Dv], lse [N]) for this request and head)."""
    if want is None:
        want = oracle.split_attention_mla(q, rows_global, DV, N, scale, base=base)
    want_o, want_lse = want[0][r], want[1][r]
    if want_lse == -np.inf:
        assert got_lse == -np.inf, f"{what}: empty rank must give lse = -inf, got {got_lse}"
        assert np.all(got_o == 0.0), f"{what}: empty rank must give O = 0"
        return 0.0
    conv = math.log(2.0) if base == "2" else 1.0
    own = rows_global[r::N]
    s = own @ q * scale                                     # natural-log units
    part = [np.r_[256 * cc:256 * cc + 256, 512 + 32 * cc:544 + 32 * cc] for cc in (0, 1)]
    s_half = sum(np.abs(own[:, cols] @ q[cols]) for cols in part)
    E = float((DK * 2.0 ** -24 * (np.abs(own) @ np.abs(q)) + 2.0 ** -11 * s_half).max()) * scale + 2.0 ** -24 * math.log(2.0)
    w = np.exp(s - want_lse * conv)
    A = w @ np.abs(own[:, :DV])
    tol_o = 2 * (u * A + u * np.abs(want_o) + 2 * E * A) + 1e-6
    err = np.abs(got_o - want_o)
    assert np.all(err <= tol_o), (f"{what}: O error {err.max():.3e} above its bound at "
                                  f"d={int(np.argmax(err - tol_o))}")
    tol_l = 2 * (E + 1e-6 * abs(want_lse * conv)) / conv + 1e-6
    assert abs(got_lse - want_lse) <= tol_l, f"{what}: lse {got_lse} vs {want_lse} (bound {tol_l:.2e})"
    return float((err / (np.abs(want_o) + 1e-3)).max())


def run(q, kv, seq, max_len, scale, base, split, o=None, lse=None):
    B, H, _ = q.shape
    N = kv.shape[0]
    if o is None:
        o = torch.full((N, B, H, DV), float("nan"), dtype=q.dtype, device=DEV)
    if lse is None:
        lse = torch.full((N, B, H), float("nan"), dtype=torch.float32, device=DEV)
    need = binding.workspace_bytes(N, B, H, DV, max_len, split)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV) if need else None
    binding.decode_attention_mla(q, kv, seq, max_len, o, lse, scale, base=base, split_tokens=split, workspace=ws)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, "a bounded wait ran out"
    return o, lse


def draw(N, B, H, lens, max_len, dtype, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    lc = (max_len + N - 1) // N
    q = torch.randn((B, H, DK), generator=g, device=DEV).to(dtype)
    kv = torch.randn((N, B, lc, DK), generator=g, device=DEV).to(dtype)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return q, kv, seq


CASES = [
    # N, H, lengths, max_len, split, dtype, base
    (2, 128, [700, 1, 130], 700, 128, torch.bfloat16, "2"),     # ragged tails, several splits
    (2, 128, [700, 1, 130], 700, 1024, torch.bfloat16, "e"),    # one split per rank
    (8, 128, [5, 64 * 8, 64 * 8 + 3, 1000], 1000, 64, torch.bfloat16, "2"),  # ranks with no token
    (4, 16, [300, 257], 300, 64, torch.float16, "e"),           # fewer heads, fp16
    (1, 128, [129, 64], 129, 1024, torch.float16, "2"),         # one rank: the whole sequence
    (3, 96, [0, 200, 1], 200, 64, torch.bfloat16, "e"),         # an empty request
]


@pytest.mark.parametrize("N,H,lens,max_len,split,dtype,base", CASES)
def test_mla_rank_partials_match_oracle_on_every_row(N, H, lens, max_len, split, dtype, base):
    B = len(lens)
    q, kv, seq = draw(N, B, H, lens, max_len, dtype, seed=N * 100 + H + split)
    scale = 192 ** -0.5
    o, lse = run(q, kv, seq, max_len, scale, base, split)
    qn = q.double().cpu().numpy()
    on = o.double().cpu().numpy()
    ln = lse.double().cpu().numpy()
    for b, L in enumerate(lens):
        rows = global_rows(kv, b, L, N)
        for h in range(H):
            want = oracle.split_attention_mla(qn[b, h], rows, DV, N, scale, base=base)
            for r in range(N):
                check_row(on[r, b, h], ln[r, b, h], qn[b, h], rows, r, N, scale, base, U[dtype],
                          f"N={N} b={b} r={r} h={h}", want)


def test_mla_stale_cache_rows_do_not_leak_into_the_result():
    # rows past a rank's local length hold whatever the cache had there (here
    # NaN and huge values): the tail tile loads them, and they must add
    # exactly nothing
    N, B, H, max_len = 2, 2, 128, 1000
    lens = [333, 77]
    q, kv, seq = draw(N, B, H, lens, max_len, torch.bfloat16, seed=31)
    clean_o, clean_lse = run(q, kv, seq, max_len, 0.07, "2", 1024)
    dirty = kv.clone()
    for r in range(N):
        for b, L in enumerate(lens):
            n_loc = L // N + (1 if r < L % N else 0)
            dirty[r, b, n_loc:, ::2] = float("nan")
            dirty[r, b, n_loc:, 1::2] = 3e38
    o, lse = run(q, dirty, seq, max_len, 0.07, "2", 1024)
    assert torch.equal(o.view(torch.int16), clean_o.view(torch.int16))
    assert torch.equal(lse, clean_lse)


def test_mla_strided_operands_give_the_contiguous_bits():
    # q sliced out of a wider projection, the cache rows padded to 640
    # elements, O rows padded and the LSE a strided slot
    N, B, H, max_len = 2, 3, 128, 400
    lens = [400, 129, 64]
    q, kv, seq = draw(N, B, H, lens, max_len, torch.bfloat16, seed=41)
    want_o, want_lse = run(q, kv, seq, max_len, 0.08, "e", 128)
    qw = torch.zeros((B, H, DK + 64), dtype=q.dtype, device=DEV)
    qw[..., 32:32 + DK] = q
    lc = kv.shape[2]
    kvw = torch.zeros((N, B, lc, 640), dtype=kv.dtype, device=DEV)
    kvw[..., :DK] = kv
    ow = torch.full((N, B, H, DV + 8), float("nan"), dtype=q.dtype, device=DEV)
    lw = torch.full((N, B, H, 2), float("nan"), dtype=torch.float32, device=DEV)
    o, lse = run(qw[..., 32:32 + DK], kvw[..., :DK], seq, max_len, 0.08, "e", 128, ow[..., :DV], lw[..., 0])
    assert torch.equal(o.view(torch.int16), want_o.view(torch.int16))
    assert torch.equal(lse, want_lse)
    assert torch.isnan(ow[..., DV:]).all() and torch.isnan(lw[..., 1]).all()


def test_mla_full_size_workload_sampled_rows():
    a = generate_mla_attention("mla_decode_attention", device=DEV)
    c = a["cfg"]
    N, B, H = c["N"], c["B"], c["H"]
    q, kv, seq, L = a["q"], a["kv"], a["seq_lens"], a["max_len"]
    o, lse = run(q, kv, seq, L, c["sm_scale"], c["base"], 1024)
    assert torch.isfinite(o.float()).all() and not torch.isnan(lse).any()
    lens = seq.cpu().tolist()
    rng = np.random.default_rng(0)
    qn = q.double().cpu().numpy()
    for _ in range(24):
        b, h, r = int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))
        rows = global_rows(kv, b, lens[b], N)
        check_row(o[r, b, h].double().cpu().numpy(), float(lse[r, b, h]), qn[b, h], rows, r, N,
                  c["sm_scale"], c["base"], U[q.dtype], f"full size b={b} r={r} h={h}")


def test_mla_schedule_leaves_every_item_bit_identical():
    """The CTA pairs are persistent and each takes its share of the (rank,
    request, split) items in turn: longest first while there are at most
    8192 items, in launch order beyond.  An item's arithmetic does not depend
    on which pair takes it or when, so a request's rows are bit for bit the
    same in a batch of 10240 items (launch order) and in a batch of that
    request alone (128 items, sorted), and they match the oracle."""
    N, H, max_len, split, B = 8, 128, 8192, 64, 80   # 8 ranks x 80 requests x 16 splits
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, max_len + 1, size=B)]
    lens[:3] = [0, max_len, 1]
    q, kv, seq = draw(N, B, H, lens, max_len, torch.bfloat16, seed=17)
    scale = 192 ** -0.5
    o, lse = run(q, kv, seq, max_len, scale, "2", split)
    for b in (0, 1, 2, 37, 79):
        o1, lse1 = run(q[b:b + 1], kv[:, b:b + 1], seq[b:b + 1], max_len, scale, "2", split)
        assert torch.equal(o1.view(torch.int16), o[:, b:b + 1].view(torch.int16)), f"request {b}: O differs"
        assert torch.equal(lse1.view(torch.int32), lse[:, b:b + 1].view(torch.int32)), f"request {b}: lse differs"
    qn = q.double().cpu().numpy()
    for b, h, r in ((1, 0, 0), (1, 127, 7), (37, 5, 3), (79, 64, 1), (2, 9, 0), (2, 9, 1)):
        rows = global_rows(kv, b, lens[b], N)
        check_row(o[r, b, h].double().cpu().numpy(), float(lse[r, b, h]), qn[b, h], rows, r, N, scale, "2",
                  U[q.dtype], f"b={b} r={r} h={h}")


def test_mla_rising_scores_move_the_reference_max_mid_item():
    """Scores that grow along the sequence make the kernel's lazily moved
    reference max move (by more than 2^8) inside items and across tiles, so
    the accumulated output is rescaled several times per item; every row
    still matches the oracle.  Several items per CTA pair (splits of 128)."""
    N, H, max_len, split = 4, 64, 3000, 128
    lens = [3000, 2500, 1700, 900, 64, 1]
    B = len(lens)
    q, kv, seq = draw(N, B, H, lens, max_len, torch.bfloat16, seed=31)
    lc = kv.shape[2]
    # local token i of rank r is global token i*N + r: scale its latent row by
    # 1 + t/300 so that later tokens score higher (the row max climbs by ~50
    # in log2 units over the longest request)
    t = torch.arange(lc, device=DEV)[None, :] * N + torch.arange(N, device=DEV)[:, None]
    kv = (kv.float() * (1.0 + t.float() / 300.0)[:, None, :, None]).to(torch.bfloat16)
    scale = 192 ** -0.5
    o, lse = run(q, kv, seq, max_len, scale, "2", split)
    qn = q.double().cpu().numpy()
    on = o.double().cpu().numpy()
    ln = lse.double().cpu().numpy()
    for b, L in enumerate(lens):
        rows = global_rows(kv, b, L, N)
        for h in (0, 17, H - 1):
            want = oracle.split_attention_mla(qn[b, h], rows, DV, N, scale, base="2")
            for r in range(N):
                check_row(on[r, b, h], ln[r, b, h], qn[b, h], rows, r, N, scale, "2", U[q.dtype],
                          f"rising scores b={b} r={r} h={h}", want)


RANDOM_SEEDS = list(range(8))


@pytest.mark.parametrize("seed", RANDOM_SEEDS)
def test_mla_random_shapes_match_oracle_on_sampled_rows(seed):
    """Seeded random shapes for the persistent kernel: 1-8 ranks, 1-40
    requests (some empty, some at the cache's end), 16-128 heads, splits of
    64 tokens to whole ranks, either payload type and LSE base; every
    request's rows for a few heads and every rank against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 9))
    B = int(rng.integers(1, 41))
    H = int(rng.choice([16, 48, 64, 96, 128]))
    max_len = int(rng.integers(1, 6001))
    split = int(rng.choice([64, 128, 512, 2048]))
    dtype = torch.bfloat16 if rng.integers(2) else torch.float16
    base = "2" if rng.integers(2) else "e"
    lens = [int(x) for x in rng.integers(0, max_len + 1, size=B)]
    lens[int(rng.integers(B))] = max_len
    if B > 2:
        lens[int(rng.integers(B))] = 0
    q, kv, seq = draw(N, B, H, lens, max_len, dtype, seed=2000 + seed)
    scale = 192 ** -0.5
    o, lse = run(q, kv, seq, max_len, scale, base, split)
    qn = q.double().cpu().numpy()
    on = o.double().cpu().numpy()
    ln = lse.double().cpu().numpy()
    heads = sorted({0, H - 1, int(rng.integers(H))})
    for b, L in enumerate(lens):
        rows = global_rows(kv, b, L, N)
        for h in heads:
            want = oracle.split_attention_mla(qn[b, h], rows, DV, N, scale, base=base)
            for r in range(N):
                check_row(on[r, b, h], ln[r, b, h], qn[b, h], rows, r, N, scale, base, U[dtype],
                          f"seed={seed} N={N} B={B} H={H} split={split} b={b} r={r} h={h}", want)


def test_whole_mla_dcp_decode_equals_unsplit_attention():
    """The one-GPU DCP decode at the MLA merge's shape (N=8 ranks, 128
    requests, 128 heads, 512 output columns, base-2 LSE): each rank's
    tensor-core attention, the peer-inside pack, the exchange as a view and
    the combine give unsplit latent attention over the whole sequence."""
    a = generate_mla_attention("mla_decode_attention", device=DEV, max_len=520)
    c = a["cfg"]
    N, B, H = c["N"], c["B"], c["H"]
    q, kv, seq, L = a["q"], a["kv"], a["seq_lens"], a["max_len"]
    o, lse = run(q, kv, seq, L, c["sm_scale"], c["base"], 64)
    H_pr = H // N
    partial_o, stats = layouts.alloc_peer_inside(N, B, H_pr, N, DV, o.dtype, DEV)
    dst_o, dst_lse = layouts.peer_inside_send_views(partial_o, stats)
    binding.pack_send(o, lse, dst_o, dst_lse)
    ro, rl = layouts.exchange_peer_inside(partial_o, stats)
    out = torch.empty((N, B, H_pr, DV), dtype=o.dtype, device=DEV)
    out_lse = torch.empty((N, B, H_pr), dtype=torch.float32, device=DEV)
    binding.lse_combine(ro, rl, out, out_lse, base=c["base"])
    torch.cuda.synchronize()
    lens = seq.cpu().tolist()
    qn = q.double().cpu().numpy()
    rng = np.random.default_rng(1)
    for _ in range(48):
        b, h = int(rng.integers(B)), int(rng.integers(H))
        rows = global_rows(kv, b, lens[b], N)
        want_o, want_lse = oracle.split_attention_mla(qn[b, h], rows, DV, 1, c["sm_scale"], base=c["base"])
        got = out[h // H_pr, b, h % H_pr].double().cpu().numpy()
        s = rows @ qn[b, h] * c["sm_scale"]
        w = np.exp(s - want_lse[0] * math.log(2.0))
        A = w @ np.abs(rows[:, :DV])
        # the attention's bound, plus one more bf16 rounding of the merged row
        tol = 3 * U[o.dtype] * (A + np.abs(want_o[0])) + 1e-5
        assert np.all(np.abs(got - want_o[0]) <= tol), f"b={b} h={h}: {np.abs(got - want_o[0]).max():.3e}"
        assert abs(float(out_lse[h // H_pr, b, h % H_pr]) - want_lse[0]) <= 1e-3


def test_mla_refuses_shapes_it_does_not_compile():
    q, kv, seq = draw(2, 1, 8, [10], 10, torch.bfloat16, seed=3)
    o = torch.empty((2, 1, 8, DV), dtype=q.dtype, device=DEV)
    lse = torch.empty((2, 1, 8), dtype=torch.float32, device=DEV)
    with pytest.raises(binding.DcpError, match="split_tokens"):
        binding.decode_attention_mla(q, kv, seq, 10, o, lse, 0.1, split_tokens=100)
    with pytest.raises(binding.DcpError, match="Dk"):
        binding.decode_attention_mla(q[..., :512], kv[..., :512], seq, 10, o, lse, 0.1)
    q3, kv3, seq3 = draw(2, 1, 130, [10], 10, torch.bfloat16, seed=4)
    o3 = torch.empty((2, 1, 130, DV), dtype=q.dtype, device=DEV)
    l3 = torch.empty((2, 1, 130), dtype=torch.float32, device=DEV)
    with pytest.raises(binding.DcpError, match="128"):
        binding.decode_attention_mla(q3, kv3, seq3, 10, o3, l3, 0.1)


# A process of its own, so that the switch that holds the loads back reaches
# no other test.
_STALL_SCRIPT = r'''
import math, os, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import oracle
from decode_context_attention_gb300 import binding

binding.load()
dev = "cuda"
g = torch.Generator(device=dev).manual_seed(5)
N, B, H, L = 2, 1, 16, 100
q = torch.randn((B, H, 576), generator=g, device=dev).to(torch.bfloat16)
kv = torch.randn((N, B, (L + N - 1) // N, 576), generator=g, device=dev).to(torch.bfloat16)
seq = torch.tensor([L], dtype=torch.int32, device=dev)
o = torch.empty((N, B, H, 512), dtype=torch.bfloat16, device=dev)
lse = torch.empty((N, B, H), dtype=torch.float32, device=dev)
scale = 192 ** -0.5
# 1: every latent-row load held back, so the first wait on them runs out
os.environ["DCP_TEST_STALL_LOADS"] = "1"
binding.decode_attention_mla(q, kv, seq, L, o, lse, scale, base="2")
torch.cuda.synchronize()
st = binding.device_status()
assert st == 7, f"expected DCP_ERR_TIMEOUT, got {st}"
assert binding.device_status() == 0, "the status must clear once read"
# 2: the context is still usable and the next call is right
del os.environ["DCP_TEST_STALL_LOADS"]
binding.decode_attention_mla(q, kv, seq, L, o, lse, scale, base="2")
torch.cuda.synchronize()
assert binding.device_status() == 0
idx = torch.arange(L, device=dev)
rows = kv[idx % N, 0, idx // N].double().cpu().numpy()
want, want_lse = oracle.split_attention_mla(q[0, 3].double().cpu().numpy(), rows, 512, N, scale, base="2")
got = o[:, 0, 3].double().cpu().numpy()
assert np.abs(got - want).max() <= 0.02 * np.abs(want).max(), np.abs(got - want).max()
assert np.abs(lse[:, 0, 3].double().cpu().numpy() - want_lse).max() <= 1e-3
print("timeout reported, context usable")
'''


def test_mla_wait_that_runs_out_reports_a_timeout_and_leaves_the_context_usable():
    # every wait of the tensor-core attention is bounded: held-back loads make
    # the first one run out (after 1 s), which must end the kernel with
    # DCP_ERR_TIMEOUT in the device status word, not hang it or fault
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.pop("DCP_TEST_STALL_LOADS", None)
    r = subprocess.run([sys.executable, "-c", _STALL_SCRIPT, root], capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "timeout reported, context usable" in r.stdout
