"""Host-side logic on CPU: the send/receive layout views the kernels are
handed (they must alias exactly the bytes the layouts name), and the seeded
workload generators (deterministic, with the structure their recipes state).
No GPU and no kernel: torch views and CPU tensors only."""
import numpy as np
import pytest
import torch

from decode_context_attention_gb300 import layouts
from decode_context_attention_gb300.workloads import WORKLOADS, generate, scaled, sweep_points


@pytest.mark.parametrize("dtype,lpd", [(torch.float32, 1), (torch.float16, 2), (torch.bfloat16, 2),
                                       (torch.float8_e4m3fn, 4)])
def test_peer_major_views_alias_payload_then_lse_word(dtype, lpd):
    S, N, B, H_pr, D = 2, 3, 2, 2, 8
    assert layouts.lse_pack_dim(dtype) == lpd
    buf = layouts.alloc_peer_major(S, N, B, H_pr, D, dtype, "cpu")
    assert buf.shape == (S, N, B, H_pr, D + lpd)
    buf.view(torch.uint8).zero_()
    pay, words = layouts.peer_major_views(buf, D)
    assert pay.shape == (S, N, B, H_pr, D) and words.shape == (S, N, B, H_pr)
    words.fill_(1.5)
    raw = buf.view(torch.uint8).reshape(S, N, B, H_pr, -1)
    e = buf.element_size()
    # the fp32 word sits right after the D payload elements of its own row
    assert torch.equal(raw[..., D * e:D * e + 4].contiguous().view(torch.float32).squeeze(-1),
                       torch.full((S, N, B, H_pr), 1.5))
    assert bool((raw[..., :D * e] == 0).all())
    # the exchange is a view: destination d's rows from source s are send[s, d]
    recv = layouts.exchange_peer_major(buf)
    assert recv.data_ptr() == buf.data_ptr() and recv.shape == (N, S, B, H_pr, D + lpd)
    assert torch.equal(layouts.materialize_peer_major(buf).view(torch.uint8), recv.contiguous().view(torch.uint8))


def test_peer_major_rejects_other_types():
    with pytest.raises(ValueError):
        layouts.lse_pack_dim(torch.float64)
    with pytest.raises(ValueError):
        layouts.lse_pack_dim(torch.int16)


def test_peer_inside_views_index_like_the_page_layout():
    S, B, H_pr, N, D = 2, 3, 2, 4, 5
    po, st = layouts.alloc_peer_inside(S, B, H_pr, N, D, torch.float32, "cpu")
    po.copy_(torch.arange(po.numel(), dtype=torch.float32).view(po.shape))
    st.copy_(torch.arange(st.numel(), dtype=torch.float32).view(st.shape))
    dst_o, dst_l = layouts.peer_inside_send_views(po, st)
    # the pack writes dst_o[s, p, b, hl] = partial_o[s, b, hl, p] and stats slot 0
    for s, p, b, hl in [(0, 0, 0, 0), (1, 3, 2, 1), (0, 2, 1, 0)]:
        assert torch.equal(dst_o[s, p, b, hl], po[s, b, hl, p])
        assert dst_l[s, p, b, hl] == st[s, b, hl, p, 0]
    ro, rl = layouts.exchange_peer_inside(po, st)
    mo, ml = layouts.materialize_peer_inside(po, st)
    # destination d merges rank s's rows partial_o[s, :, :, d]
    for d, s in [(0, 0), (3, 1), (2, 0)]:
        assert torch.equal(ro[d, s], po[s, :, :, d]) and torch.equal(rl[d, s], st[s, :, :, d, 0])
        assert torch.equal(mo[d, s], po[s, :, :, d]) and torch.equal(ml[d, s], st[s, :, :, d, 0])
    # slot 1 is never part of a view the kernels write or read
    assert dst_l.stride()[-1] == 2 * N and ro.shape == (N, S, B, H_pr, D)


def test_generators_are_deterministic_and_keep_their_structure():
    w = scaled(WORKLOADS["mha_decode"], B=20)
    a, b = generate(w, "cpu"), generate(w, "cpu")
    assert torch.equal(a["o"].view(torch.int16), b["o"].view(torch.int16)) and torch.equal(a["lse"], b["lse"])
    emp = a["empty"]
    k = round(0.1 * w.B)                                       # empty tokens drawn per rank
    assert w.N * k - w.B <= int(emp.sum()) <= w.N * k          # less any orphan handed back to rank 0
    assert bool((emp.sum(0) < w.N).all())                      # every token keeps an owner
    assert bool((a["lse"][emp] == -float("inf")).all()) and bool((a["o"][emp] == 0).all())
    assert bool(((a["lse"][~emp] >= 0) & (a["lse"][~emp] <= 12)).all())
    c = generate(scaled(w, seed=w.seed + 1), "cpu")
    assert not torch.equal(a["lse"], c["lse"])


def test_sweep_recipe_spread_and_fp8_payloads():
    pts = sweep_points()
    assert len(pts) == 48 and len({p.name for p in pts}) == 48 and len({p.seed for p in pts}) == 48
    w = scaled([p for p in pts if p.N == 8][0], B=16)
    d = generate(w, "cpu")
    spread = d["lse"].amax(0) - d["lse"].amin(0)
    assert bool((spread <= 40.0 + 1e-4).all()) and float(spread.max()) > 1.0
    f = generate(scaled(WORKLOADS["mla_decode_fp8"], B=4), "cpu")
    assert f["o"].dtype == torch.float8_e4m3fn
    vals = f["o"].float()
    assert bool(torch.isfinite(vals).all()) and float(vals.abs().max()) <= 448.0


def test_cached_extend_injects_the_stated_fraction_of_specials():
    w = scaled(WORKLOADS["cached_extend"], B=32)
    d = generate(w, "cpu")
    o, lse = d["o"], d["lse"]
    k_o = int(round(1e-4 * o.numel()))
    bad_o = int((~torch.isfinite(o)).sum())
    assert 0 < bad_o <= k_o                                    # drawn with replacement
    kinds = {float(x) for x in o[~torch.isfinite(o)].tolist() if not np.isnan(x)}
    assert kinds <= {float("inf"), -float("inf")}
