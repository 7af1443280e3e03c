"""Buffers and views of the two DCP send layouts and of the exchange model.

Only allocation and stride bookkeeping lives here (torch views); the data
movement is done by the CUDA kernels behind the C ABI.

Notation: S source ranks, N peers (destination ranks), B tokens, H_pr = H / N
heads per peer, D head dim, lpd = payload elements per fp32 LSE word.

* Peer-major interleaved send buffer (one flat buffer for a single
  all-to-all, split by byte offset; sglang PR #34651 report, "实现拆解" item 2):
  ``send[s] : [N, B, H_pr, D + lpd]``; payload view ``[..., :D]``, LSE view =
  the fp32 word at word index D // lpd of each row.
* Peer-inside split layout (sglang PR #34651 report, "关键源码片段",
  `_dcp_fi_a2a_lse_reduce`): ``partial_o[s] : [B, H_pr, N, D]``,
  ``stats[s] : [B, H_pr, N, 2]`` fp32 with slot 1 never written; the pack
  writes through ``partial_o.permute(2,0,1,3)`` and
  ``stats[..., 0].permute(2,0,1)``.
* Exchange model: with all S = N ranks stacked on one device, the all-to-all
  that gives destination d the peer-d block of every source is a view of the
  sender stack with the source and peer axes swapped (zero bytes moved).
  ``materialize_*`` builds the contiguous receive buffer a real all-to-all
  would have produced, for tests that want that exact layout.
"""
from __future__ import annotations

import torch


def lse_pack_dim(dtype: torch.dtype) -> int:
    """Payload elements one fp32 word occupies: 1 for fp32, 2 for 16-bit types,
    4 for fp8 e4m3."""
    if dtype not in (torch.float32, torch.float16, torch.bfloat16, torch.float8_e4m3fn):
        raise ValueError(f"no interleaved layout for {dtype}")
    return 4 // torch.empty((), dtype=dtype).element_size()


# ---- peer-major interleaved ----------------------------------------------------

def alloc_peer_major(S: int, N: int, B: int, H_pr: int, D: int, dtype, device) -> torch.Tensor:
    """Send stack [S, N, B, H_pr, D + lpd] (uninitialised)."""
    return torch.empty((S, N, B, H_pr, D + lse_pack_dim(dtype)), dtype=dtype, device=device)


def peer_major_views(buf: torch.Tensor, D: int):
    """(payload view [..., :D], fp32 LSE word view) of an interleaved buffer."""
    lpd = lse_pack_dim(buf.dtype)
    words = buf.view(torch.float32)
    return buf[..., :D], words[..., D // lpd]


def exchange_peer_major(send: torch.Tensor) -> torch.Tensor:
    """Receive rows for every destination: recv[d, s] = send[s, d] (a view)."""
    return send.transpose(0, 1)


def materialize_peer_major(send: torch.Tensor) -> torch.Tensor:
    return exchange_peer_major(send).contiguous()


# ---- peer-inside split ----------------------------------------------------------

def alloc_peer_inside(S: int, B: int, H_pr: int, N: int, D: int, dtype, device):
    """(partial_o [S, B, H_pr, N, D], stats [S, B, H_pr, N, 2] fp32), uninitialised."""
    partial_o = torch.empty((S, B, H_pr, N, D), dtype=dtype, device=device)
    stats = torch.empty((S, B, H_pr, N, 2), dtype=torch.float32, device=device)
    return partial_o, stats


def peer_inside_send_views(partial_o: torch.Tensor, stats: torch.Tensor):
    """The pack's destinations [S, N, B, H_pr, D] and [S, N, B, H_pr]."""
    return partial_o.permute(0, 3, 1, 2, 4), stats[..., 0].permute(0, 3, 1, 2)


def exchange_peer_inside(partial_o: torch.Tensor, stats: torch.Tensor):
    """Combine inputs per destination: o[d, s] = partial_o[s, :, :, d], lse likewise (views)."""
    return partial_o.permute(3, 0, 1, 2, 4), stats[..., 0].permute(3, 0, 1, 2)


def materialize_peer_inside(partial_o: torch.Tensor, stats: torch.Tensor):
    """The receive buffers a real all-to-all produces per destination d:
    o_out[d] : [B, H_pr, S, D] and stats_out[d] : [B, H_pr, S, 2], returned as
    the combine's views [d, s, B, H_pr, D] / [d, s, B, H_pr]."""
    o_out = partial_o.permute(3, 1, 2, 0, 4).contiguous()
    stats_out = stats.permute(3, 1, 2, 0, 4).contiguous()
    return o_out.permute(0, 3, 1, 2, 4), stats_out[..., 0].permute(0, 3, 1, 2)
