"""Pins for the fp64 CPU oracle (CPU only, no GPU).

Each test checks the oracle against something other than itself: numpy /
torch decoding and index maps, closed forms derived by hand, invariants the
pages state (identity at one rank, neutral empty ranks, round-robin partition
properties), the semantics of the torch routines the pages' merge calls, and
brute force (single-query softmax attention split across ranks by the
round-robin owner rule, then merged, equals unsplit attention).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def page_cases():
    with open(os.path.join(GOLDEN, "page_cases.json")) as f:
        return json.load(f)


def rand_bits(rng, shape, dtype):
    """Random payload bit patterns (any bits, NaN payloads included)."""
    if dtype == "f32":
        return rng.integers(0, 2**32, size=shape, dtype=np.uint32).view(np.float32)
    if dtype == "fp8":
        return rng.integers(0, 2**8, size=shape, dtype=np.uint8)
    bits = rng.integers(0, 2**16, size=shape, dtype=np.uint16)
    return bits.view(np.float16) if dtype == "f16" else bits


def as_u8(a):
    return np.ascontiguousarray(a).view(np.uint8)


# --------------------------------------------------------------------------
# element decoding
# --------------------------------------------------------------------------

def test_f16_decoder_matches_numpy_on_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("f16", bits.view(np.float16))
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decoder_matches_torch_on_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("bf16", bits)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_fp8_e4m3_decoder_matches_torch_on_every_bit_pattern():
    bits = np.arange(256, dtype=np.uint32).astype(np.uint8)
    got = oracle.decode("fp8", bits)
    want = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(want)
    assert nan.sum() == 2  # 0x7f and 0xff; e4m3fn has no infinities
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_lse_pack_dim():
    # vLLM #41160, "实现拆解" item 2: fp16 -> 2, fp32 -> 1; bf16 is the other
    # 16-bit output type and takes 2 as well.  The page notes that fp8 is
    # rejected there; this library extends it: an fp32 word is four fp8 elements.
    assert oracle.lse_pack_dim("f32") == 1
    assert oracle.lse_pack_dim("f16") == 2
    assert oracle.lse_pack_dim("bf16") == 2
    assert oracle.lse_pack_dim("fp8") == 4
    assert oracle.lse_pack_dim("int4") == -1


# --------------------------------------------------------------------------
# pack: both layouts, bit-exact against numpy index maps
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sentinel", [0.0, -12345.5])
def test_pack_peer_inside_matches_page_layout(sentinel):
    """sglang #34651 `test_pack_serves_the_split_peer_inside_layout`: the shapes
    the page tests, bf16 payload; expected = out.view(B,N,Hpr,D).permute(0,2,1,3)."""
    rng = np.random.default_rng(1)
    for N, B, Hpr, D in page_cases()["peer_inside_pack_shapes"]["value"]:
        H = Hpr * N
        out = rand_bits(rng, (B, H, D), "bf16")
        lse = rng.standard_normal((B, H)).astype(np.float32)
        partial_o = np.full((B, Hpr, N, D), 0xA5A5, dtype=np.uint16)
        stats = np.full((B, Hpr, N, 2), sentinel, dtype=np.float32)
        oracle.pack("bf16", N, out[None], lse[None],
                    partial_o.transpose(2, 0, 1, 3)[None], stats[..., 0].transpose(2, 0, 1)[None])
        want_o = out.reshape(B, N, Hpr, D).transpose(0, 2, 1, 3)
        want_lse = lse.reshape(B, N, Hpr).transpose(0, 2, 1)
        assert np.array_equal(as_u8(partial_o), as_u8(want_o))
        assert np.array_equal(as_u8(stats[..., 0]), as_u8(want_lse))
        # slot 1 is never written
        assert np.array_equal(stats[..., 1], np.full_like(stats[..., 1], sentinel))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "fp8"])
@pytest.mark.parametrize("pad", [0, 3])
def test_pack_peer_major_interleaved_bytes(dtype, pad):
    """sglang #34651 "实现拆解" item 2 / vLLM #41160: send buffer [N,B,Hpr,D+lpd];
    payload view [..., :D], fp32 word view at word D//lpd.  With `pad` extra
    elements per row, the padding must keep its sentinel bytes."""
    rng = np.random.default_rng(2)
    lpd = oracle.lse_pack_dim(dtype)
    e = {"f32": 4, "fp8": 1}.get(dtype, 2)
    for N, B, H, D in [(2, 4, 16, 128), (4, 3, 8, 12), (1, 2, 4, 8), (8, 2, 8, 64)]:
        Hpr = H // N
        out = rand_bits(rng, (B, H, D), dtype)
        lse = rand_bits(rng, (B, H), "f32")
        W = D + lpd + (lpd * pad)
        send = np.empty((N, B, Hpr, W), dtype=out.dtype)
        send.view(np.uint8)[...] = 0x5A
        words = send.view(np.float32)  # [N,B,Hpr,W*e/4]
        oracle.pack(dtype, N, out[None], lse[None], send[..., :D][None], words[..., D // lpd][None])
        payload = as_u8(out.reshape(B, N, Hpr, D).transpose(1, 0, 2, 3)).reshape(N, B, Hpr, D * e)
        lseb = as_u8(lse.reshape(B, N, Hpr).transpose(1, 0, 2)).reshape(N, B, Hpr, 4)
        padb = np.full((N, B, Hpr, pad * lpd * e), 0x5A, dtype=np.uint8)
        want = np.concatenate([payload, lseb, padb], axis=-1)
        assert np.array_equal(send.view(np.uint8).reshape(N, B, Hpr, W * e), want)


def test_pack_groups_and_strided_source():
    """G source ranks in one call; source O read through a transposed view."""
    rng = np.random.default_rng(3)
    G, N, B, H, D = 3, 4, 5, 8, 16
    Hpr = H // N
    base = rand_bits(rng, (B, G, H, D), "f16")
    o = base.transpose(1, 0, 2, 3)  # [G,B,H,D], strided
    lse_base = rand_bits(rng, (H, B, G), "f32")
    lse = lse_base.transpose(2, 1, 0)  # [G,B,H], strided
    dst = np.zeros((G, B, Hpr, N, D), dtype=np.float16)
    stats = np.zeros((G, B, Hpr, N, 2), dtype=np.float32)
    oracle.pack("f16", N, o, lse, dst.transpose(0, 3, 1, 2, 4), stats[..., 0].transpose(0, 3, 1, 2))
    for g in range(G):
        want = o[g].reshape(B, N, Hpr, D).transpose(0, 2, 1, 3)
        assert np.array_equal(as_u8(dst[g]), as_u8(want))
        assert np.array_equal(as_u8(stats[g, ..., 0]), as_u8(lse[g].reshape(B, N, Hpr).transpose(0, 2, 1)))


def test_pack_rejects_heads_not_divisible():
    o = np.zeros((1, 2, 6, 4), dtype=np.float32)
    lse = np.zeros((1, 2, 6), dtype=np.float32)
    dst = np.zeros((1, 4, 2, 1, 4), dtype=np.float32)
    dl = np.zeros((1, 4, 2, 1), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.pack("f32", 4, o, lse, dst, dl)


# --------------------------------------------------------------------------
# combine: closed forms
# --------------------------------------------------------------------------

def stack(os_, lses, dtype=np.float32):
    """[N, D] rows and [N] LSEs -> oracle views [G=1, N, B=1, Hc=1, D] / [1, N, 1, 1]."""
    o = np.asarray(os_, dtype=dtype)[None, :, None, None, :]
    l = np.asarray(lses, dtype=np.float32)[None, :, None, None]
    return o, l


def test_two_rank_worked_example_base2():
    # base-2 LSEs (0, 1): weights 2^0 : 2^1 = 1/3 : 2/3
    # out = (1*[3,6,-3] + 2*[0,3,6]) / 3 = [1, 4, 3];  global LSE = log2(1 + 2)
    o, l = stack([[3, 6, -3], [0, 3, 6]], [0.0, 1.0])
    out, G = oracle.combine("f32", o, l, base="2")
    assert np.allclose(out.ravel(), [1.0, 4.0, 3.0], rtol=0, atol=1e-14)
    assert abs(G.item() - math.log2(3.0)) < 1e-14


def test_three_rank_worked_example_base2():
    # LSEs (1, 1, 2) base 2: weights 2 : 2 : 4 over 8 = 1/4, 1/4, 1/2
    # out = 4/4 + 8/4 + 2/2 = 4;  global LSE = log2(8) = 3
    o, l = stack([[4.0], [8.0], [2.0]], [1.0, 1.0, 2.0])
    out, G = oracle.combine("f32", o, l, base="2")
    assert abs(out.item() - 4.0) < 1e-14
    assert abs(G.item() - 3.0) < 1e-14


def test_two_rank_closed_form_base_e():
    rng = np.random.default_rng(4)
    for _ in range(50):
        l = rng.uniform(-6, 6, size=2).astype(np.float32)
        O = rng.standard_normal((2, 7))
        o, lv = stack(O, l, dtype=np.float64)
        out, G = oracle.combine("f64", o, lv, base="e")
        a, b = math.exp(float(l[0])), math.exp(float(l[1]))
        want = (a * O[0] + b * O[1]) / (a + b)
        assert np.allclose(out.ravel(), want, rtol=1e-13, atol=1e-13)
        assert abs(G.item() - math.log(a + b)) < 1e-13


# --------------------------------------------------------------------------
# combine: invariants
# --------------------------------------------------------------------------

def test_single_rank_is_identity_including_non_finite():
    """sglang #34213: world_size == 1 returns (out, lse) unchanged."""
    O = np.array([[1.5, np.nan, np.inf, -2.0]], dtype=np.float32)
    for lse in (0.25, -np.inf, np.nan, np.inf):
        o, l = stack(O, [lse])
        for sanitize in (False, True):
            out, G = oracle.combine("f32", o, l, sanitize=sanitize)
            assert np.array_equal(out.ravel(), O.ravel().astype(np.float64), equal_nan=True)
            assert np.array_equal(G.ravel(), np.array([lse]), equal_nan=True)


def test_neutral_empty_ranks_are_bit_exact():
    """A rank owning no KV, given as (0, -inf), leaves every output bit unchanged
    wherever it is inserted (sglang #33926, `fixup_zero_kv_rows`)."""
    rng = np.random.default_rng(5)
    for N in (1, 2, 3, 5):
        O = rng.standard_normal((N, 9)).astype(np.float32)
        l = rng.uniform(-5, 5, size=N).astype(np.float32)
        if N == 1:
            ref_out, ref_G = O[0].astype(np.float64), np.float64(l[0])
        else:
            o, lv = stack(O, l)
            ref_out, ref_G = oracle.combine("f32", o, lv)
        for pos in range(N + 1):
            O2 = np.insert(O, pos, 0.0, axis=0)
            l2 = np.insert(l, pos, -np.inf)
            o, lv = stack(O2, l2)
            out, G = oracle.combine("f32", o, lv)
            assert np.array_equal(out.ravel(), np.ravel(ref_out))
            assert np.array_equal(G.ravel(), np.ravel(ref_G))


def test_shift_invariance():
    rng = np.random.default_rng(6)
    O = rng.standard_normal((4, 16))
    l = rng.integers(-192, 192, size=4) / 64.0  # shifts below stay exact in fp32
    for c in (-50.0, -1.0, 0.5, 30.0):
        o0, l0 = stack(O, l, dtype=np.float64)
        o1, l1 = stack(O, (l + c), dtype=np.float64)
        # the shift must be exact in fp32 for the comparison to be fair
        assert np.array_equal(l1.astype(np.float64) - l0.astype(np.float64), np.full(l1.shape, c))
        out0, G0 = oracle.combine("f64", o0, l0)
        out1, G1 = oracle.combine("f64", o1, l1)
        assert np.allclose(out0, out1, rtol=0, atol=1e-12)
        assert abs((G1 - G0).item() - c) < 1e-12


def test_base2_agrees_with_base_e_after_conversion():
    rng = np.random.default_rng(7)
    O = rng.standard_normal((6, 11))
    le = rng.uniform(0, 12, size=6).astype(np.float32)
    l2 = (le.astype(np.float64) / math.log(2.0)).astype(np.float32)
    out_e, G_e = oracle.combine("f64", *stack(O, le, dtype=np.float64), base="e")
    out_2, G_2 = oracle.combine("f64", *stack(O, l2, dtype=np.float64), base="2")
    # only the fp32 rounding of the converted LSEs separates the two
    assert np.allclose(out_e, out_2, rtol=0, atol=1e-5)
    assert abs(G_2.item() * math.log(2.0) - G_e.item()) < 1e-5


def test_rank_order_does_not_matter():
    rng = np.random.default_rng(8)
    O = rng.standard_normal((8, 5))
    l = rng.uniform(0, 20, size=8).astype(np.float32)
    out, G = oracle.combine("f64", *stack(O, l, dtype=np.float64))
    perm = rng.permutation(8)
    out_p, G_p = oracle.combine("f64", *stack(O[perm], l[perm], dtype=np.float64))
    assert np.allclose(out, out_p, rtol=0, atol=1e-13)
    assert abs(G.item() - G_p.item()) < 1e-13


def test_weights_underflow_at_spread_40():
    """LSE spread of 40 (base e) makes the small ranks' weights ~e^-40, not 0 or NaN."""
    O = np.array([[1.0], [1e17]])
    l = np.array([40.0, 0.0], dtype=np.float32)
    out, G = oracle.combine("f64", *stack(O, l, dtype=np.float64))
    w1 = math.exp(-40.0) / (1 + math.exp(-40.0))
    assert abs(out.item() - ((1 - w1) * 1.0 + w1 * 1e17)) < 1e-6


# --------------------------------------------------------------------------
# combine: non-finite LSE and O (reading of torch logsumexp + nan_to_num)
# --------------------------------------------------------------------------

def test_non_finite_lse_classes():
    O = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], dtype=np.float32)
    # any NaN -> global NaN, every weight NaN -> 0, out = 0
    out, G = oracle.combine("f32", *stack(O, [1.0, np.nan, 2.0]))
    assert np.isnan(G.item()) and np.array_equal(out.ravel(), [0.0, 0.0])
    # any +inf -> global +inf, weights 0 (finite ranks) or NaN->0 (the +inf rank)
    out, G = oracle.combine("f32", *stack(O, [1.0, np.inf, 2.0]))
    assert G.item() == np.inf and np.array_equal(out.ravel(), [0.0, 0.0])
    # NaN wins over +inf
    out, G = oracle.combine("f32", *stack(O, [np.inf, np.nan, 2.0]))
    assert np.isnan(G.item())
    # all ranks empty -> global -inf, out = 0
    out, G = oracle.combine("f32", *stack(np.zeros((3, 2)), [-np.inf] * 3))
    assert G.item() == -np.inf and np.array_equal(out.ravel(), [0.0, 0.0])


def test_non_finite_o_with_and_without_sanitize():
    O = np.array([[np.nan, 2.0, np.inf], [3.0, -np.inf, 5.0]], dtype=np.float32)
    l = [0.0, 0.0]  # equal weights 1/2
    out, _ = oracle.combine("f32", *stack(O, l), sanitize=True)
    assert np.array_equal(out.ravel(), [1.5, 1.0, 2.5])
    out, _ = oracle.combine("f32", *stack(O, l), sanitize=False)
    assert np.isnan(out[..., 0]).all() and out[..., 1].item() == -np.inf
    assert out[..., 2].item() == np.inf


def test_agrees_with_torch_semantics_of_the_ag_rs_merge():
    """sglang #34213 `cp_lse_ag_out_rs_mha`: torch.logsumexp over the stacked LSE,
    exp(lse - global), nan_to_num(scale), nan_to_num_(O), multiply, sum over ranks.
    Run in fp64 on CPU on inputs with injected NaN/+-inf."""
    rng = np.random.default_rng(9)
    N, T, H, D = 4, 6, 5, 8
    O = rng.standard_normal((N, T, H, D)).astype(np.float32)
    L = rng.uniform(0, 15, size=(N, T, H)).astype(np.float32)
    specials = np.array([np.nan, np.inf, -np.inf], dtype=np.float32)
    O.reshape(-1)[rng.choice(O.size, 40, replace=False)] = rng.choice(specials, 40)
    L.reshape(-1)[rng.choice(L.size, 12, replace=False)] = rng.choice(specials, 12)
    L[:, 0, 0] = -np.inf  # an all-empty row
    lses = torch.from_numpy(L).double()
    glob = torch.logsumexp(lses, dim=0)
    scale = torch.nan_to_num(torch.exp(lses - glob).unsqueeze(-1), nan=0.0, posinf=0.0, neginf=0.0)
    o_t = torch.nan_to_num(torch.from_numpy(O).double(), nan=0.0, posinf=0.0, neginf=0.0)
    want = (o_t * scale).sum(0).numpy()
    out, G = oracle.combine("f32", O[None], L[None], sanitize=True)
    assert np.allclose(out[0], want, rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.isnan(G[0]), np.isnan(glob.numpy()))
    fin = np.isfinite(glob.numpy())
    assert np.array_equal(G[0][~fin & ~np.isnan(G[0])], glob.numpy()[~fin & ~np.isnan(G[0])])
    assert np.allclose(G[0][fin], glob.numpy()[fin], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# brute force: split attention + merge == unsplit attention
# --------------------------------------------------------------------------

def full_attention(q, K, V, scale):
    s = (K @ q) * scale
    m = s.max()
    p = np.exp(s - m)
    lse = m + math.log(p.sum())
    return (p / p.sum()) @ V, lse


def test_dcp_lens_page_invariants():
    """sglang #33926 `TestDcpDecodeLayout`: per-rank lengths sum to the global
    length; appending one token grows exactly rank (L-1) % n; and the count
    matches brute force over the owner rule t % n."""
    cases = page_cases()["dcp_layout"]["value"]
    for n in cases["sizes"]:
        for L in range(0, cases["max_len"] + 1):
            lens = [oracle.dcp_lens(L, n, r) for r in range(n)]
            assert sum(lens) == L
            assert lens == [sum(1 for t in range(L) if t % n == r) for r in range(n)]
            if L >= 1:
                grew = [lens[r] - oracle.dcp_lens(L - 1, n, r) for r in range(n)]
                assert sum(grew) == 1 and grew[(L - 1) % n] == 1


def test_split_attention_single_rank_is_full_attention():
    rng = np.random.default_rng(10)
    for L in (1, 2, 7, 40):
        D = 5
        q, K, V = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
        O, lse = oracle.split_attention(q, K, V, 1, 0.5)
        want, want_lse = full_attention(q, K, V, 0.5)
        assert np.allclose(O[0], want, rtol=0, atol=1e-13)
        assert abs(lse[0] - want_lse) < 1e-13
        O2, lse2 = oracle.split_attention(q, K, V, 1, 0.5, base="2")
        assert abs(lse2[0] * math.log(2.0) - want_lse) < 1e-13


def test_split_attention_ranks_without_tokens_are_neutral_pairs():
    rng = np.random.default_rng(11)
    q, K, V = rng.standard_normal(3), rng.standard_normal((2, 3)), rng.standard_normal((2, 3))
    O, lse = oracle.split_attention(q, K, V, 5, 1.0)
    for r in range(2, 5):
        assert lse[r] == -np.inf and np.array_equal(O[r], np.zeros(3))
    # rank r alone sees only token r: O_r = V_r and lse_r = score_r
    for r in range(2):
        assert np.allclose(O[r], V[r], atol=1e-15)
        assert abs(lse[r] - float(K[r] @ q)) < 1e-14


@pytest.mark.parametrize("base", ["e", "2"])
def test_merged_split_attention_equals_unsplit_attention(base):
    """Many independent (g, b, h) attention problems, each split over N ranks by
    the round-robin owner rule, merged through a strided [G,N,B,Hc,D] view."""
    rng = np.random.default_rng(12 if base == "e" else 13)
    G, B, Hc, D = 2, 3, 5, 4
    for N in page_cases()["dcp_layout"]["value"]["sizes"]:
        buf = np.zeros((B, N, Hc, G, D))          # storage order differs from view order
        lbuf = np.zeros((Hc, G, B, N), dtype=np.float32)
        want = np.zeros((G, B, Hc, D))
        want_lse = np.zeros((G, B, Hc))
        for g in range(G):
            for b in range(B):
                for h in range(Hc):
                    L = int(rng.integers(1, 41))
                    q, K, V = (rng.standard_normal(D), rng.standard_normal((L, D)),
                               rng.standard_normal((L, D)))
                    O, lse = oracle.split_attention(q, K, V, N, 0.7, base=base)
                    buf[b, :, h, g, :] = O
                    lbuf[h, g, b, :] = lse
                    want[g, b, h], want_lse[g, b, h] = full_attention(q, K, V, 0.7)
        o = buf.transpose(3, 1, 0, 2, 4)    # [G,N,B,Hc,D]
        lv = lbuf.transpose(1, 3, 2, 0)     # [G,N,B,Hc]
        out, G_ = oracle.combine("f64", o, lv, base=base)
        # fp32 rounding of the per-rank LSE bounds the agreement
        assert np.allclose(out, want, rtol=0, atol=2e-6)
        conv = math.log(2.0) if base == "2" else 1.0
        assert np.allclose(G_ * conv, want_lse, rtol=0, atol=2e-6)


def latent_attention(q, KV, Dv, scale):
    """Unsplit single-query attention over latent rows: scores over the whole
    row, the value is the row's first Dv elements (numpy, for the pins)."""
    return full_attention(q, KV, KV[:, :Dv], scale)


def test_split_attention_mla_single_rank_is_full_latent_attention():
    # one rank owns every token: attention over the whole latent cache, the
    # value being each row's first Dv elements; a nonzero rope part moves the
    # scores, not the value
    rng = np.random.default_rng(14)
    for L in (1, 2, 9, 40):
        Dk, Dv = 12, 8
        q, KV = rng.standard_normal(Dk), rng.standard_normal((L, Dk))
        O, lse = oracle.split_attention_mla(q, KV, Dv, 1, 0.4)
        want, want_lse = latent_attention(q, KV, Dv, 0.4)
        assert np.allclose(O[0], want, rtol=0, atol=1e-13)
        assert abs(lse[0] - want_lse) < 1e-13
        O2, lse2 = oracle.split_attention_mla(q, KV, Dv, 1, 0.4, base="2")
        assert np.array_equal(O2, O)
        assert abs(lse2[0] * math.log(2.0) - want_lse) < 1e-13
        # the rope columns enter only through the scores
        KV2 = KV.copy()
        KV2[:, Dv:] = 0.0
        q2 = q.copy()
        q2[Dv:] = 0.0
        O3, lse3 = oracle.split_attention_mla(q2, KV2, Dv, 1, 0.4)
        want3, want3_lse = full_attention(q[:Dv], KV[:, :Dv], KV[:, :Dv], 0.4)
        assert np.allclose(O3[0], want3, rtol=0, atol=1e-13) and abs(lse3[0] - want3_lse) < 1e-13


def test_split_attention_mla_at_full_value_width_is_split_attention():
    # with Dv = Dk the latent row is both key and value: the MHA split
    # attention with K = V = KV, rank by rank, for every group size
    rng = np.random.default_rng(15)
    for n in page_cases()["dcp_layout"]["value"]["sizes"]:
        for L in (0, 1, 3, 17):
            D = 6
            q, KV = rng.standard_normal(D), rng.standard_normal((L, D))
            O, lse = oracle.split_attention_mla(q, KV, D, n, 0.9, base="2")
            O2, lse2 = oracle.split_attention(q, KV, KV, n, 0.9, base="2")
            assert np.allclose(O, O2, rtol=0, atol=1e-14)
            fin = np.isfinite(lse2)
            assert np.array_equal(np.isfinite(lse), fin) and np.all(lse[~fin] == -np.inf)
            assert np.allclose(lse[fin], lse2[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("base", ["e", "2"])
def test_merged_split_attention_mla_equals_unsplit_attention(base):
    """Split over N ranks by the round-robin owner rule and merged by the
    combine, latent-cache attention equals unsplit attention (numpy)."""
    rng = np.random.default_rng(16 if base == "e" else 17)
    Dk, Dv = 10, 6
    for N in page_cases()["dcp_layout"]["value"]["sizes"]:
        for L in range(1, 41, 3):
            q, KV = rng.standard_normal(Dk), rng.standard_normal((L, Dk))
            O, lse = oracle.split_attention_mla(q, KV, Dv, N, 0.6, base=base)
            for r in range(N):
                assert (lse[r] == -np.inf) == (r >= L)
            out, G_ = oracle.combine("f64", O[None, :, None, None, :],
                                     lse.astype(np.float32)[None, :, None, None], base=base)
            want, want_lse = latent_attention(q, KV, Dv, 0.6)
            assert np.allclose(out[0, 0, 0], want, rtol=0, atol=2e-6)
            conv = math.log(2.0) if base == "2" else 1.0
            assert abs(G_[0, 0, 0] * conv - want_lse) < 2e-6


# --------------------------------------------------------------------------
# fused unpack + combine over the interleaved receive rows
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "fp8"])
def test_unpack_combine_equals_combine_on_separated_views(dtype):
    rng = np.random.default_rng(14)
    lpd = oracle.lse_pack_dim(dtype)
    G, N, B, Hpr, D = 2, 4, 3, 5, 16
    if dtype == "bf16":
        vals = torch.randn(G, N, B, Hpr, D, dtype=torch.bfloat16)
        payload = vals.view(torch.int16).numpy().view(np.uint16)
    elif dtype == "fp8":
        vals = torch.randn(G, N, B, Hpr, D).to(torch.float8_e4m3fn)
        payload = vals.view(torch.uint8).numpy()
    else:
        payload = rng.standard_normal((G, N, B, Hpr, D)).astype(np.float16 if dtype == "f16" else np.float32)
    lse = rng.uniform(-3, 9, size=(G, N, B, Hpr)).astype(np.float32)
    lse[0, 1, 2, :] = -np.inf
    recv = np.zeros((G, N, B, Hpr, D + lpd), dtype=payload.dtype)
    recv[..., :D] = payload
    recv.view(np.float32)[..., D // lpd] = lse
    for base in ("e", "2"):
        out_u, G_u = oracle.unpack_combine(dtype, recv, D, base=base)
        out_c, G_c = oracle.combine(dtype, recv[..., :D], recv.view(np.float32)[..., D // lpd], base=base)
        assert np.array_equal(out_u, out_c) and np.array_equal(G_u, G_c)


def test_unpack_combine_brute_force_through_interleaved_rows():
    rng = np.random.default_rng(15)
    N, D = 3, 8
    B = 6
    recv = np.zeros((1, N, B, 1, D + 1), dtype=np.float32)
    want = np.zeros((B, D))
    for b in range(B):
        L = int(rng.integers(1, 12))
        q, K, V = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
        O, lse = oracle.split_attention(q, K, V, N, 0.3)
        recv[0, :, b, 0, :D] = O
        recv[0, :, b, 0, D] = lse
        want[b] = full_attention(q, K, V, 0.3)[0]
    out, _ = oracle.unpack_combine("f32", recv, D)
    assert np.allclose(out[0, :, 0, :], want, rtol=0, atol=5e-6)


def test_unpack_combine_single_rank_is_identity():
    recv = np.zeros((1, 1, 2, 2, 6), dtype=np.float16)
    recv[..., :4] = np.array([1.0, np.nan, -np.inf, 3.0], dtype=np.float16)
    recv.view(np.float32)[..., 2] = np.array([[-np.inf, 1.0], [np.nan, 7.5]], dtype=np.float32)
    out, G = oracle.unpack_combine("f16", recv, 4)
    assert np.array_equal(out[0], recv[0, 0, ..., :4].astype(np.float64), equal_nan=True)
    assert np.array_equal(G[0], recv.view(np.float32)[0, 0, ..., 2].astype(np.float64), equal_nan=True)
