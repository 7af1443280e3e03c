"""Seeded synthetic inputs for the DCP merge workloads.

This module only *draws* inputs: per-rank partial attention outputs O and
their log-sum-exp values, stacked over the N ranks of one decode-context-
parallel group, plus the structure the pages describe (ranks that own no KV
for a token, NaN/inf injection).  It holds none of the merge arithmetic, so
both the CUDA path and the CPU oracle can be fed from it.

Workloads (shapes and value distributions follow the pages' decode and
cached-extend cases; no model weights or datasets are involved):

  tiny           N=2, B=4, H=16, D=128, fp32 O ~ N(0,1), LSE ~ U(-5,5) base e;
                 one (rank, token) pair is empty: O = 0 and LSE = -inf on every
                 head.  Peer-major pack + combine.
  mha_decode     N=4, B=64, H=32, D=128, bf16 O ~ N(0,1), LSE ~ U(0,12) base e;
                 per rank round(0.1*B) tokens are empty, every token keeps at
                 least one owning rank.  Peer-major pack + fused unpack+combine.
  mla_decode     N=8, B=128, H=128, D=512 (absorbed-MLA kv_lora_rank), bf16 O,
                 LSE ~ U(0,20) base 2.  Peer-inside pack + combine over the
                 strided receive views.
  sweep          N in {2,4,8} x B in {1,8,32,256} x D in {128,512}, H=64, fp16 O,
                 base-e LSE l_r = c + s*u_r with c ~ U(0,12), s ~ U(0,40) per
                 (token, head) and u_r ~ U(0,1) per rank (max - min up to 40);
                 both pack layouts (48 points).
  mla_decode_fp8 the MLA decode shape (N=8, B=128, H=128, D=512) with fp8 e4m3
                 O (N(0,1) drawn in fp32, rounded to e4m3), LSE ~ U(0,20) base 2,
                 peer-major interleaved rows (lpd = 4).  Pack + fused
                 unpack+combine.
  cached_extend  N=8, T=16384, H=96, D=512, fp32 O ~ N(0,1) (3 GiB per rank),
                 LSE ~ U(0,15) base e; round(1e-4 * numel) positions of O and of
                 the LSE, drawn uniformly with replacement, are set to NaN, +inf
                 or -inf with equal odds.  In-place combine + head slices.

  mha_decode_attention  the step before the merge: N=4 ranks, B=64 requests,
                 H=32 query heads over 32 KV heads, D=128, bf16; request lengths
                 ~ U(1, 16384); every rank's local K/V cache holds its
                 round-robin share (local token i of rank r = global token
                 i*N + r), values ~ N(0,1); queries ~ N(0,1).
  gqa_decode_attention  the same with grouped-query heads: 32 query heads
                 over 4 KV heads (8 per KV head), seed 7.
  mla_decode_attention  the attention whose partials the MLA decode merge
                 takes (DeepSeek-V3-like absorbed MLA): N=8 ranks, B=128
                 requests, H=128 query heads over one latent row per token of
                 576 = 512 (kv_lora_rank, the value) + 64 (rope) bf16
                 elements, base-2 LSE, request lengths ~ U(1, 16384), latent
                 rows and absorbed queries ~ N(0,1), sm_scale = 1/sqrt(192)
                 (the no-rope plus rope query width of that model), seed 8.

An empty (rank, token) pair is the pages' neutral state for a rank that owns
no KV slice of that request: O = 0, LSE = -inf (sglang PR #33926 report,
"实现拆解" item 3, `fixup_zero_kv_rows`).  KV ownership is per token, so the
pair covers every head.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
                "fp8": torch.float8_e4m3fn}


@dataclass(frozen=True)
class Workload:
    name: str
    N: int          # ranks in the DCP group
    B: int          # tokens (decode batch, or cached-extend tokens T)
    H: int          # query heads
    D: int          # head dim of O (v_head_dim or kv_lora_rank)
    dtype: str      # payload type of O: "f32" | "f16" | "bf16" | "fp8"
    base: str       # LSE base: "e" | "2"
    layout: str     # "peer_major" | "peer_inside" | "inplace"
    kind: str       # value recipe, one of the module docstring's workloads
    seed: int

    @property
    def H_pr(self) -> int:
        return self.H // self.N


WORKLOADS = {
    "tiny": Workload("tiny", 2, 4, 16, 128, "f32", "e", "peer_major", "tiny", 0),
    "mha_decode": Workload("mha_decode", 4, 64, 32, 128, "bf16", "e", "peer_major", "mha_decode", 1),
    "mla_decode": Workload("mla_decode", 8, 128, 128, 512, "bf16", "2", "peer_inside", "mla_decode", 2),
    "mla_decode_fp8": Workload("mla_decode_fp8", 8, 128, 128, 512, "fp8", "2", "peer_major", "mla_decode", 6),
    "cached_extend": Workload("cached_extend", 8, 16384, 96, 512, "f32", "e", "inplace",
                              "cached_extend", 4),
}


def sweep_points() -> list[Workload]:
    """The 48 long-context decode sweep points (24 shapes x 2 pack layouts)."""
    pts = []
    i = 0
    for layout in ("peer_major", "peer_inside"):
        for N in (2, 4, 8):
            for B in (1, 8, 32, 256):
                for D in (128, 512):
                    pts.append(Workload(f"sweep_{layout}_N{N}_B{B}_D{D}", N, B, 64, D, "f16", "e",
                                        layout, "sweep", 3000 + i))
                    i += 1
    return pts


def scaled(w: Workload, **kw) -> Workload:
    """Same recipe at other sizes (for small parity cases)."""
    return replace(w, **kw)


def _uniform(shape, lo, hi, g, device):
    return torch.empty(shape, dtype=torch.float32, device=device).uniform_(lo, hi, generator=g)


def _normal_payload(N, B, H, D, dtype, g, device):
    o = torch.empty((N, B, H, D), dtype=TORCH_DTYPES[dtype], device=device)
    for r in range(N):  # one rank at a time keeps the fp32 temporaries small
        if o.element_size() == 1:   # fp8: draw in fp32, round once
            o[r].copy_(torch.empty((B, H, D), device=device).normal_(generator=g))
        else:
            o[r].normal_(generator=g)
    return o


def _empty_pairs(mask_nb, o, lse):
    """Apply the neutral (O = 0, LSE = -inf) state to the (rank, token) pairs in mask_nb."""
    idx = mask_nb.nonzero(as_tuple=True)
    o.view(torch.uint8)[idx] = 0    # all-zero bytes are +0 in every payload type
    lse[idx] = float("-inf")


def _inject(t, frac, g, device):
    n = t.numel()
    k = int(round(frac * n))
    if k == 0:
        return
    pos = torch.randint(0, n, (k,), generator=g, device=device)
    which = torch.randint(0, 3, (k,), generator=g, device=device)
    specials = torch.tensor([float("nan"), float("inf"), float("-inf")], device=device,
                            dtype=t.dtype)
    t.view(-1)[pos] = specials[which]


def generate(w: Workload, device="cuda", seed: int | None = None) -> dict:
    """Draw the stacked per-rank inputs of workload `w`.

    Returns {"o": [N,B,H,D] payload tensor, "lse": [N,B,H] fp32 tensor,
    "empty": [N,B] bool (True where the rank owns no KV for the token)}.
    """
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    N, B, H, D = w.N, w.B, w.H, w.D
    o = _normal_payload(N, B, H, D, w.dtype, g, device)
    empty = torch.zeros((N, B), dtype=torch.bool, device=device)
    if w.kind == "tiny":
        lse = _uniform((N, B, H), -5.0, 5.0, g, device)
        r = int(torch.randint(0, N, (1,), generator=g, device=device).item())
        b = int(torch.randint(0, B, (1,), generator=g, device=device).item())
        empty[r, b] = True
    elif w.kind == "mha_decode":
        lse = _uniform((N, B, H), 0.0, 12.0, g, device)
        k = int(round(0.1 * B))
        for r in range(N):
            perm = torch.randperm(B, generator=g, device=device)
            empty[r, perm[:k]] = True
        orphan = empty.all(dim=0)           # keep at least one owner per token
        empty[0, orphan] = False
    elif w.kind == "mla_decode":
        lse = _uniform((N, B, H), 0.0, 20.0, g, device)
    elif w.kind == "sweep":
        c = _uniform((1, B, H), 0.0, 12.0, g, device)
        s = _uniform((1, B, H), 0.0, 40.0, g, device)
        u = _uniform((N, 1, 1), 0.0, 1.0, g, device)
        lse = c + s * u
    elif w.kind == "cached_extend":
        lse = _uniform((N, B, H), 0.0, 15.0, g, device)
        _inject(o, 1e-4, g, device)
        _inject(lse, 1e-4, g, device)
    else:
        raise ValueError(f"unknown workload kind {w.kind!r}")
    if bool(empty.any()):
        _empty_pairs(empty, o, lse)
    return {"o": o, "lse": lse, "empty": empty}


ATTENTION = {"mha_decode_attention": dict(N=4, B=64, H=32, Hkv=32, D=128, dtype="bf16", max_len=16384,
                                          base="e", seed=5),
             "gqa_decode_attention": dict(N=4, B=64, H=32, Hkv=4, D=128, dtype="bf16", max_len=16384,
                                          base="e", seed=7)}


def generate_attention(name="mha_decode_attention", device="cuda", seed=None, **override) -> dict:
    """Draw a decode-attention workload: q [B,H,D], each rank's local caches
    k, v [N,B,Lc,Hkv,D] (Lc = ceil(max_len / N); entries past a rank's local
    length are never read), seq_lens [B] int32 global lengths in [1, max_len]."""
    c = dict(ATTENTION[name], **override)
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(c["seed"] if seed is None else seed)
    N, B, H, Hkv, D, L = c["N"], c["B"], c["H"], c["Hkv"], c["D"], c["max_len"]
    dt = TORCH_DTYPES[c["dtype"]]
    lc = (L + N - 1) // N
    q = torch.empty((B, H, D), dtype=dt, device=device).normal_(generator=g)
    k = torch.empty((N, B, lc, Hkv, D), dtype=dt, device=device)
    v = torch.empty((N, B, lc, Hkv, D), dtype=dt, device=device)
    for r in range(N):
        k[r].normal_(generator=g)
        v[r].normal_(generator=g)
    seq = torch.randint(1, L + 1, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    return {"q": q, "k": k, "v": v, "seq_lens": seq, "max_len": L, "cfg": c}


MLA_ATTENTION = {"mla_decode_attention": dict(N=8, B=128, H=128, Dk=576, Dv=512, dtype="bf16", max_len=16384,
                                              base="2", seed=8, sm_scale=192 ** -0.5)}


def generate_mla_attention(name="mla_decode_attention", device="cuda", seed=None, **override) -> dict:
    """Draw an absorbed-MLA decode workload: q [B,H,Dk], each rank's latent
    cache kv [N,B,Lc,Dk] (Lc = ceil(max_len / N); local token i of rank r is
    global token i*N + r; entries past a rank's local length are never
    used), seq_lens [B] int32 global lengths in [1, max_len]."""
    c = dict(MLA_ATTENTION[name], **override)
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(c["seed"] if seed is None else seed)
    N, B, H, Dk, L = c["N"], c["B"], c["H"], c["Dk"], c["max_len"]
    dt = TORCH_DTYPES[c["dtype"]]
    lc = (L + N - 1) // N
    q = torch.empty((B, H, Dk), dtype=dt, device=device).normal_(generator=g)
    kv = torch.empty((N, B, lc, Dk), dtype=dt, device=device)
    for r in range(N):
        kv[r].normal_(generator=g)
    seq = torch.randint(1, L + 1, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    return {"q": q, "kv": kv, "seq_lens": seq, "max_len": L, "cfg": c}
