#!/usr/bin/env python3
"""Benchmark of the DCP LSE merge on GB300: µs per call and achieved HBM GB/s.

Default workload (one "call" = one step): the MLA decode merge, N = 8 ranks,
B = 128 tokens, H = 128 heads, D = 512 (absorbed-MLA kv_lora_rank), bf16
partial outputs, base-2 LSE.  One step is the whole hot path for all 8 ranks
held on one GPU: the peer-inside pack of every source rank (one launch, G = 8)
followed by the LSE combine for every destination rank (one launch, G = 8)
over the receive views; the all-to-all between them is a zero-copy view of
the sender stack.  L2 is flushed before every kernel (a 2x-L2 write, then a
2x-L2 read so no dirty lines are left), outside the timed events, so every
kernel reads its inputs from HBM.

Also measured in the same run and reported under "secondary":
  * one rank's own calls of the headline workload (G = 1: the pack of one
    source, the combine of one destination);
  * the two-collective layout at the largest long-context sweep point (N = 8,
    B = 256, H = 64, D = 512, fp16): O and LSE packed into separate buffers,
    combine without a returned LSE;
  * the same sweep point through the interleaved pack and the fused
    unpack+combine;
  * the MLA decode shape with fp8 e4m3 payloads through the interleaved pack
    (lpd = 4) and the fused unpack+combine;
  * the decode attention that produces the merge's inputs (N = 4 ranks,
    B = 64 requests, H = 32, D = 128, bf16, lengths up to 16384): one query
    head per KV head (MHA, ~9 GB of K/V, CUDA cores), and 8 per KV head (GQA,
    ~1.1 GB, tcgen05), the latter also over 64-token pages;
  * the absorbed-MLA decode attention whose outputs the headline merge takes
    (N = 8, B = 128, H = 128, 576-wide latent rows, 512-wide values, bf16, on
    the tcgen05 tensor cores), in TFLOP/s and GB/s;
  * the cached-extend workload (N = 8, 16384 tokens, 96 heads, D = 512, fp32;
    29 GB per call): the combine writing the per-rank head slices
    contiguously, then the in-place sanitising combine.

`--impl reference` times the fp64 CPU oracle instead, on a bounded sample of
the same workload, and reports it in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DCP LSE-merge µs/call and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
UNIT = "µs/call"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic bytes (what each call must move, whatever the implementation)
# ---------------------------------------------------------------------------

def bytes_pack(G, B, H, D, e):
    """Read O and LSE of G*B*H rows, write the same bytes to the send layout."""
    return 2 * G * B * H * (D * e + 4)


def bytes_merge(G, N, B, Hc, D, e, return_lse=True):
    """Read N rank rows (payload + LSE word) per output row, write the row (+ LSE)."""
    rows = G * B * Hc
    return N * rows * (D * e + 4) + rows * D * e + (rows * 4 if return_lse else 0)


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU under torchrun; weak scaling)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def max_over_ranks(x: float, device=None) -> float:
    """Max of a host float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# clocks (nvidia-smi sampled while the GPU works)
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        samples = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                samples.append((float(parts[0]), float(parts[1]), float(parts[2]),
                                float(parts[3]), parts[4:8]))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s in samples if s[3] > 0] or samples
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in busy for i, v in enumerate(s[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[0] for s in busy),
                "sm_max_mhz": max(s[1] for s in samples),
                "power_w_max": max(s[2] for s in samples),
                "reasons": reasons, "samples": len(samples), "samples_busy": len(busy)}


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------

class L2Flush:
    """Evict L2 between timed launches: write one buffer of 2x L2, then read a
    second one, so L2 ends up holding clean lines of neither the inputs nor the
    flush (a write-only flush would leave dirty lines whose write-back the next
    timed kernel would pay for)."""

    def __init__(self, device):
        import torch

        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 64 << 20)
        self.wbuf = torch.empty(n, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(n // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.wbuf.zero_()
        self.rbuf.amax()

    def evict(self):
        """Read a third 2x-L2 buffer: every line in L2 is replaced, and the
        dirty ones are written back to HBM on the way."""
        if not hasattr(self, "ebuf"):
            import torch

            self.ebuf = torch.zeros_like(self.rbuf)
        self.ebuf.amax()


def time_with_writeback(launch, steps, warmup, flush, device):
    """Time of `launch` including the HBM write-back of the lines it leaves
    dirty in L2.  A kernel's stores can still sit in L2 when its end event
    fires; here an eviction pass follows it inside the timed region, and the
    same pass over a clean L2 (timed separately) is subtracted.  Returns
    (mean ms with write-back, mean ms of the eviction pass alone)."""
    import torch

    def bracket(with_kernel):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush()
        e0.record()
        if with_kernel:
            launch()
        flush.evict()
        e1.record()
        return e0, e1

    for _ in range(warmup):
        bracket(True)
        bracket(False)
    torch.cuda.synchronize(device)
    ev = [(bracket(True), bracket(False)) for _ in range(steps)]
    torch.cuda.synchronize(device)
    with_k = statistics.fmean(a.elapsed_time(b) for (a, b), _ in ev)
    alone = statistics.fmean(a.elapsed_time(b) for _, (a, b) in ev)
    return with_k - alone, alone


def time_sequence(launches, steps, warmup, flush, device):
    """Run `steps` iterations of the launch sequence; before each launch flush
    L2 (unless flush is None), bracket each launch with CUDA events on the
    current stream.  Returns per-launch lists of durations in ms."""
    import torch

    for _ in range(warmup):
        for f in launches:
            if flush:
                flush()
            f()
    torch.cuda.synchronize(device)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in launches] for _ in range(steps)]
    barrier(device)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(steps):
        for j, f in enumerate(launches):
            if flush:
                flush()
            ev[i][j][0].record()
            f()
            ev[i][j][1].record()
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    barrier(device)
    per = [[ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(steps)] for j in range(len(launches))]
    return per, wall


def kernel_record(name, ms_list, nbytes, peak_gbs):
    avg = statistics.fmean(ms_list)
    gbs = nbytes / (avg * 1e-3) / 1e9
    return {"kernel": name, "us_per_launch": round(avg * 1e3, 3),
            "us_median": round(statistics.median(ms_list) * 1e3, 3),
            "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak_gbs, 4)}


def theoretical_hbm_gbs(gpu_index: int):
    """Nominal DRAM bandwidth from the driver's read-only queries: 2 transfers
    per memory clock x bus width.  None where NVML is not available."""
    import ctypes

    try:
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            return None
        try:
            dev = ctypes.c_void_p()
            if nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(dev)) != 0:
                return None
            mhz, bits = ctypes.c_uint(), ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(dev, ctypes.c_int(2), ctypes.byref(mhz)) != 0:  # memory clock
                return None
            if nvml.nvmlDeviceGetMemoryBusWidth(dev, ctypes.byref(bits)) != 0:
                return None
            return round(2 * mhz.value * 1e6 * bits.value / 8 / 1e9, 1)
        finally:
            nvml.nvmlShutdown()
    except (OSError, AttributeError):
        return None


def load_tensor_peak():
    """Dense bf16 tensor throughput (TFLOP/s) for a kernel timed on its own:
    the burst figure of MEASURED_PEAKS.json, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
    return 1900.0, "fallback"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# The source files that define each profiled kernel's code: a counter taken on
# a kernel stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "pack_kernel": ("dcp_pack.cu", "dcp_device.cuh"),
    "combine_kernel": ("dcp_combine.cuh", "dcp_combine_bf16.cu", "dcp_device.cuh"),
    "decode_partial_kernel": ("dcp_attention.cu", "dcp_device.cuh"),
    "decode_partial_mma_kernel": ("dcp_attention.cu", "dcp_device.cuh"),
    "gqa_decode_tc_kernel": ("dcp_attention_tc.cu", "dcp_device.cuh", "dcp_sm100.cuh"),
    "mla_decode_kernel": ("dcp_mla_attention.cu", "dcp_device.cuh", "dcp_sm100.cuh"),
}


def csrc_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "decode_context_attention_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """dram read+write bytes per launch from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get("kernels", {}).get(kernel)
    if not ent or kernel not in KERNEL_SOURCES or ent.get("csrc_digest") != csrc_digest(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# the workloads as launch sequences
# ---------------------------------------------------------------------------

def setup_mla_decode(device, seed_offset=0):
    import torch

    from decode_context_attention_gb300 import binding, layouts
    from decode_context_attention_gb300.workloads import WORKLOADS, generate, scaled

    w = WORKLOADS["mla_decode"]
    if seed_offset:
        w = scaled(w, seed=w.seed + 100 * seed_offset)
    d = generate(w, device)
    S, B, H, D = d["o"].shape
    N, H_pr = w.N, w.H_pr
    partial_o, stats = layouts.alloc_peer_inside(S, B, H_pr, N, D, d["o"].dtype, device)
    dst_o, dst_lse = layouts.peer_inside_send_views(partial_o, stats)
    ro, rl = layouts.exchange_peer_inside(partial_o, stats)
    out = torch.empty((N, B, H_pr, D), dtype=d["o"].dtype, device=device)
    out_lse = torch.empty((N, B, H_pr), dtype=torch.float32, device=device)
    pack = binding.prepare_pack_send(d["o"], d["lse"], dst_o, dst_lse)
    comb = binding.prepare_lse_combine(ro, rl, out, out_lse, base=w.base)
    e = d["o"].element_size()
    return {
        "w": w, "d": d, "out": out, "out_lse": out_lse, "partial_o": partial_o, "stats": stats,
        "launches": [pack, comb],
        "names": ["dcp_pack_send (peer-inside, G=8 sources)",
                  "dcp_lse_combine (strided recv views, G=8 destinations)"],
        "kernels": ["pack_kernel", "combine_kernel"],
        "bytes": [bytes_pack(S, B, H, D, e), bytes_merge(N, S, B, H_pr, D, e)],
    }


def setup_cached_extend(device, tokens=None, slices=False):
    import torch

    from decode_context_attention_gb300 import binding
    from decode_context_attention_gb300.workloads import WORKLOADS, generate, scaled

    w = WORKLOADS["cached_extend"]
    if tokens:
        w = scaled(w, B=tokens)
    d = generate(w, device)
    o, lse = d["o"], d["lse"]
    N, T, H, D = o.shape
    out_lse = torch.empty((T, H), dtype=torch.float32, device=device)
    comb = binding.prepare_lse_combine(o, lse, o[0], out_lse, base=w.base, sanitize=True,
                                       inplace=True)
    if not slices:
        return {"w": w, "launches": [comb], "keep": (o, lse, out_lse),
                "names": ["dcp_lse_combine (in place, sanitise, fp32)"],
                "bytes": [bytes_merge(1, N, T, H, D, 4)]}
    # the per-rank head slices [k*H/N, (k+1)*H/N) written contiguously by the
    # combine itself (group axis = slice), from the same inputs
    hs = H // N
    o_k = o.view(N, T, N, hs, D).permute(2, 0, 1, 3, 4)
    l_k = lse.view(N, T, N, hs).permute(2, 0, 1, 3)
    sl = torch.empty((N, T, hs, D), dtype=o.dtype, device=device)
    sl_lse = torch.empty((N, T, hs), dtype=torch.float32, device=device)
    slc = binding.prepare_lse_combine(o_k, l_k, sl, sl_lse, base=w.base, sanitize=True)
    return {"w": w, "launches": [slc, comb], "keep": (o, lse, out_lse, sl, sl_lse),
            "names": ["dcp_lse_combine (contiguous head slices, sanitise, fp32)",
                      "dcp_lse_combine (in place, sanitise, fp32)"],
            "bytes": [bytes_merge(1, N, T, H, D, 4)] * 2}


def page_pools(k, v, page_size, seed=0):
    """Each rank's local caches [N, B, Lc, Hkv, D] moved into a page pool
    [N, B * max_pages, page_size, Hkv, D] in a shuffled page order, with the
    page table [N, B, max_pages] int32 that finds them."""
    import torch

    N, B, Lc, Hkv, D = k.shape
    max_pages = (Lc + page_size - 1) // page_size
    g = torch.Generator().manual_seed(seed)
    bt = torch.stack([torch.randperm(B * max_pages, generator=g) for _ in range(N)]).to(k.device)
    pools = []
    for src in (k, v):
        pool = torch.empty((N, B * max_pages, page_size, Hkv, D), dtype=src.dtype, device=src.device)
        for r in range(N):
            pad = torch.zeros((B, max_pages * page_size, Hkv, D), dtype=src.dtype, device=src.device)
            pad[:, :Lc] = src[r]
            pool[r, bt[r]] = pad.view(B * max_pages, page_size, Hkv, D)
        pools.append(pool)
    return pools[0], pools[1], bt.view(N, B, max_pages).to(torch.int32)


def setup_decode_attention(device, split_tokens=1024, batch=None, name="mha_decode_attention", page_size=0):
    import math

    import torch

    from decode_context_attention_gb300 import binding
    from decode_context_attention_gb300.workloads import generate_attention

    a = generate_attention(name, device=device, **({"B": batch} if batch else {}))
    c = a["cfg"]
    N, B, H, Hkv, D = c["N"], c["B"], c["H"], c["Hkv"], c["D"]
    o = torch.empty((N, B, H, D), dtype=a["q"].dtype, device=device)
    lse = torch.empty((N, B, H), dtype=torch.float32, device=device)
    nbytes = binding.workspace_bytes(N, B, H, D, a["max_len"], split_tokens)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device) if nbytes else None
    if page_size:
        kp, vp, bt = page_pools(a["k"], a["v"], page_size)
        del a["k"], a["v"]
        a["k_pages"], a["v_pages"], a["block_table"] = kp, vp, bt
        call = binding.prepare_decode_attention_paged(a["q"], kp, vp, bt, a["seq_lens"], a["max_len"], o, lse,
                                                      1.0 / math.sqrt(D), base=c["base"],
                                                      split_tokens=split_tokens, workspace=ws)
    else:
        call = binding.prepare_decode_attention(a["q"], a["k"], a["v"], a["seq_lens"], a["max_len"], o, lse,
                                                1.0 / math.sqrt(D), base=c["base"], split_tokens=split_tokens,
                                                workspace=ws)
    tokens = int(a["seq_lens"].sum().item())
    e = a["q"].element_size()
    # K and V rows of every owned token, each rank's read of q, O and LSE written
    algo = 2 * tokens * Hkv * D * e + N * B * H * D * e + N * B * H * D * e + N * B * H * 4
    return {"launches": [call], "keep": (a, o, lse, ws), "tokens": tokens, "workspace_bytes": nbytes,
            "name": name,
            "names": [f"dcp_decode_attention{'_paged' if page_size else ''} (N={N} B={B} H={H} Hkv={Hkv} "
                      f"D={D} bf16, {tokens} KV tokens, splits of {split_tokens}"
                      f"{f', {page_size}-token pages' if page_size else ''})"],
            "bytes": [algo]}


def setup_mla_attention(device, split_tokens=2048, batch=None, max_len=None):
    """Each rank's absorbed-MLA decode attention (the step whose outputs the
    MLA decode merge takes), on the tensor cores."""
    import torch

    from decode_context_attention_gb300 import binding
    from decode_context_attention_gb300.workloads import generate_mla_attention

    over = {}
    if batch:
        over["B"] = batch
    if max_len:
        over["max_len"] = max_len
    a = generate_mla_attention("mla_decode_attention", device=device, **over)
    c = a["cfg"]
    N, B, H, Dk, Dv = c["N"], c["B"], c["H"], c["Dk"], c["Dv"]
    o = torch.empty((N, B, H, Dv), dtype=a["q"].dtype, device=device)
    lse = torch.empty((N, B, H), dtype=torch.float32, device=device)
    nbytes = binding.workspace_bytes(N, B, H, Dv, a["max_len"], split_tokens)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device) if nbytes else None
    call = binding.prepare_decode_attention_mla(a["q"], a["kv"], a["seq_lens"], a["max_len"], o, lse,
                                                c["sm_scale"], base=c["base"], split_tokens=split_tokens,
                                                workspace=ws)
    tokens = int(a["seq_lens"].sum().item())
    e = a["q"].element_size()
    # every owned latent row once, each rank's read of q, O and LSE written
    algo = tokens * Dk * e + N * B * H * Dk * e + N * B * H * Dv * e + N * B * H * 4
    flops = 2 * tokens * H * (Dk + Dv)  # scores over Dk, value product over Dv, every head
    return {"launches": [call], "keep": (a, o, lse, ws), "tokens": tokens, "workspace_bytes": nbytes,
            "flops": flops,
            "names": [f"dcp_decode_attention_mla (N={N} B={B} H={H} Dk={Dk} Dv={Dv} bf16, {tokens} latent "
                      f"rows, splits of {split_tokens})"],
            "bytes": [algo]}


def setup_sweep_max(device):
    from decode_context_attention_gb300.workloads import sweep_points

    w = [p for p in sweep_points() if p.layout == "peer_major" and p.N == 8 and p.B == 256
         and p.D == 512][0]
    return setup_peer_major(w, device)


def setup_mla_fp8(device):
    from decode_context_attention_gb300.workloads import WORKLOADS

    return setup_peer_major(WORKLOADS["mla_decode_fp8"], device)


def setup_two_collective(device):
    """The legacy two-collective layout at the largest sweep point: O and LSE
    packed into separate peer-major buffers (one all-to-all each), then the
    combine over the exchanged views without a returned LSE."""
    import torch

    from decode_context_attention_gb300 import binding
    from decode_context_attention_gb300.workloads import generate, sweep_points

    w = [p for p in sweep_points() if p.layout == "peer_major" and p.N == 8 and p.B == 256
         and p.D == 512][0]
    d = generate(w, device)
    S, B, H, D = d["o"].shape
    N, H_pr = w.N, w.H_pr
    send_o = torch.empty((S, N, B, H_pr, D), dtype=d["o"].dtype, device=device)
    send_l = torch.empty((S, N, B, H_pr), dtype=torch.float32, device=device)
    out = torch.empty((N, B, H_pr, D), dtype=d["o"].dtype, device=device)
    pack = binding.prepare_pack_send(d["o"], d["lse"], send_o, send_l)
    comb = binding.prepare_lse_combine(send_o.transpose(0, 1), send_l.transpose(0, 1), out, None,
                                       base=w.base)
    e = d["o"].element_size()
    return {"w": w, "launches": [pack, comb], "keep": (d, send_o, send_l, out),
            "names": [f"dcp_pack_send (separate O and LSE buffers, G={S})",
                      f"dcp_lse_combine (separate recv views, no returned LSE, G={N})"],
            "bytes": [bytes_pack(S, B, H, D, e), bytes_merge(N, S, B, H_pr, D, e, return_lse=False)]}


def setup_per_rank(device):
    """One rank's own calls of the MLA decode merge (G = 1): the pack of source
    0 and the combine of destination 0."""
    import torch

    from decode_context_attention_gb300 import binding, layouts
    from decode_context_attention_gb300.workloads import WORKLOADS, generate

    w = WORKLOADS["mla_decode"]
    d = generate(w, device)
    S, B, H, D = d["o"].shape
    N, H_pr = w.N, w.H_pr
    partial_o, stats = layouts.alloc_peer_inside(S, B, H_pr, N, D, d["o"].dtype, device)
    dst_o, dst_lse = layouts.peer_inside_send_views(partial_o, stats)
    binding.pack_send(d["o"], d["lse"], dst_o, dst_lse)
    # destination 0 merges its own receive buffer, as a real all-to-all leaves
    # it: o_out [B, H_pr, N, D] and stats [B, H_pr, N, 2], contiguous
    ro, rl = layouts.materialize_peer_inside(partial_o, stats)
    ro, rl = ro[:1].clone(), rl[:1]
    out = torch.empty((1, B, H_pr, D), dtype=d["o"].dtype, device=device)
    out_lse = torch.empty((1, B, H_pr), dtype=torch.float32, device=device)
    pack = binding.prepare_pack_send(d["o"][:1], d["lse"][:1], dst_o[:1], dst_lse[:1])
    comb = binding.prepare_lse_combine(ro, rl, out, out_lse, base=w.base)
    e = d["o"].element_size()
    return {"w": w, "launches": [pack, comb], "keep": (d, partial_o, stats, ro, rl, out, out_lse),
            "names": ["dcp_pack_send (peer-inside, one source rank, G=1)",
                      "dcp_lse_combine (one destination rank, G=1)"],
            "bytes": [bytes_pack(1, B, H, D, e), bytes_merge(1, N, B, H_pr, D, e)]}


def setup_peer_major(w, device):
    """Interleaved pack of every source rank, then the fused unpack+combine of
    every destination over the exchanged rows (a view of the send stack)."""
    import torch

    from decode_context_attention_gb300 import binding, layouts
    from decode_context_attention_gb300.workloads import generate

    d = generate(w, device)
    S, B, H, D = d["o"].shape
    N, H_pr = w.N, w.H_pr
    send = layouts.alloc_peer_major(S, N, B, H_pr, D, d["o"].dtype, device)
    pay, words = layouts.peer_major_views(send, D)
    binding.pack_send(d["o"], d["lse"], pay, words)
    recv = layouts.exchange_peer_major(send)
    out = torch.empty((N, B, H_pr, D), dtype=d["o"].dtype, device=device)
    out_lse = torch.empty((N, B, H_pr), dtype=torch.float32, device=device)
    pack = binding.prepare_pack_send(d["o"], d["lse"], pay, words)
    fused = binding.prepare_unpack_combine(recv, D, out, out_lse, base=w.base)
    e = d["o"].element_size()
    return {"w": w, "launches": [pack, fused], "keep": (d, send, out, out_lse), "d": d, "send": send,
            "names": [f"dcp_pack_send (peer-major interleaved, G={S})",
                      f"dcp_unpack_combine (interleaved recv, G={N})"],
            "bytes": [bytes_pack(S, B, H, D, e), bytes_merge(N, S, B, H_pr, D, e)]}


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle_units(unit, threads: int, budget_s: float):
    """Run oracle work units on `threads` host threads until `budget_s` has
    passed.  unit(k) processes the k-th independent share of a call (other
    ranks' rows for other k; the oracle's arithmetic is unchanged, and its C
    calls release the GIL) and returns the fraction of a call it covered.
    Returns (seconds, calls done)."""
    from concurrent.futures import ThreadPoolExecutor

    stop = time.perf_counter() + budget_s

    def worker(i):
        done, k = 0.0, i
        while True:
            done += unit(k)
            k += threads
            if time.perf_counter() >= stop:
                return done

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        done = sum(ex.map(worker, range(threads)))
    return time.perf_counter() - t0, done


def host_payload(t):
    """Contiguous host copy of a payload tensor in the oracle's representation."""
    import numpy as np
    import torch

    t = t.detach().contiguous().cpu()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_host_inputs(mla):
    """Host copies of every source rank's pack inputs and every destination
    rank's combine inputs of the MLA decode workload."""
    d = mla["d"]
    o = host_payload(d["o"])                                 # [S, B, H, D]
    lse = d["lse"].detach().contiguous().cpu().numpy()       # [S, B, H]
    po = host_payload(mla["partial_o"])                      # [S, B, H_pr, N, D]
    st = mla["stats"][..., 0].contiguous().cpu().numpy()     # [S, B, H_pr, N]
    return mla["w"], o, lse, po, st


def oracle_mla_unit(inputs, k, b0=0, b1=None):
    """Share k of an MLA decode call through the oracle: source rank s = k % N
    packs its partials and destination rank s merges what it receives
    (partial_o[:, :, :, s] of every source), over tokens [b0, b1) (all by
    default).  Returns the fraction of a call processed."""
    import numpy as np

    import oracle

    w, o, lse, po, st = inputs
    N, H_pr, D = w.N, w.H_pr, w.D
    s = k % N
    b1 = o.shape[1] if b1 is None else b1
    nb = b1 - b0
    dst = np.empty((nb, H_pr, N, D), dtype=np.uint16)
    stats = np.zeros((nb, H_pr, N, 2), dtype=np.float32)
    oracle.pack("bf16", N, o[s:s + 1, b0:b1], lse[s:s + 1, b0:b1], dst.transpose(2, 0, 1, 3)[None],
                stats[..., 0].transpose(2, 0, 1)[None])
    oracle.combine("bf16", po[None, :, b0:b1, :, s], st[None, :, b0:b1, :, s], base=w.base)
    return (nb / w.B) / N


def time_oracle(mla, budget_s: float, threads: int):
    """Oracle µs per full MLA decode call on `threads` host threads."""
    inputs = oracle_host_inputs(mla)
    el, done = run_oracle_units(lambda k: oracle_mla_unit(inputs, k), threads, budget_s)
    return el / done * 1e6, el, done


def time_oracle_attention(at, budget_s: float, threads: int):
    """Oracle µs per decode-attention call: sampled (request, head) rows of the
    workload through oracle.split_attention (every rank at once) on `threads`
    host threads, scaled by the KV tokens of the whole call."""
    import numpy as np
    import torch

    import oracle

    a = at["keep"][0]
    c = a["cfg"]
    N, H, Hkv, D = c["N"], c["H"], c["Hkv"], c["D"]
    lens = a["seq_lens"].cpu().tolist()
    rng = np.random.default_rng(0)
    total = at["tokens"] * H  # every (token, query head) pair of the call
    samples = []
    for _ in range(2 * threads):
        b, h = int(rng.integers(len(lens))), int(rng.integers(H))
        L = lens[b]
        idx = torch.arange(L, device=a["k"].device)
        hk = h // (H // Hkv)
        kg = a["k"][idx % N, b, idx // N, hk].double().cpu().numpy()
        vg = a["v"][idx % N, b, idx // N, hk].double().cpu().numpy()
        samples.append((a["q"][b, h].double().cpu().numpy(), kg, vg, L))

    def unit(k):
        q, kg, vg, L = samples[k % len(samples)]
        oracle.split_attention(q, kg, vg, N, 1.0 / D ** 0.5, base=c["base"])
        return L / total

    el, done = run_oracle_units(unit, threads, budget_s)
    return el / done * 1e6, el, done


def time_oracle_mla_attention(at, budget_s: float, threads: int):
    """Oracle µs per MLA decode-attention call: sampled (request, head) rows
    through oracle.split_attention_mla (every rank at once) on `threads` host
    threads, scaled by the latent rows of the whole call."""
    import numpy as np
    import torch

    import oracle

    a = at["keep"][0]
    c = a["cfg"]
    N, H, Dv = c["N"], c["H"], c["Dv"]
    lens = a["seq_lens"].cpu().tolist()
    rng = np.random.default_rng(0)
    total = at["tokens"] * H
    samples = []
    for _ in range(2 * threads):
        b, h = int(rng.integers(len(lens))), int(rng.integers(H))
        L = lens[b]
        idx = torch.arange(L, device=a["kv"].device)
        rows = a["kv"][idx % N, b, idx // N].double().cpu().numpy()
        samples.append((a["q"][b, h].double().cpu().numpy(), rows, L))

    def unit(k):
        q, rows, L = samples[k % len(samples)]
        oracle.split_attention_mla(q, rows, Dv, N, c["sm_scale"], base=c["base"])
        return L / total

    el, done = run_oracle_units(unit, threads, budget_s)
    return el / done * 1e6, el, done


def time_oracle_cached_extend(budget_s: float, threads: int):
    """Oracle µs per cached-extend call from a small all-rows sample (the same
    recipe at 64 tokens) on `threads` host threads, scaled by the row count."""
    import oracle
    from decode_context_attention_gb300.workloads import WORKLOADS, generate, scaled

    w = WORKLOADS["cached_extend"]
    small = scaled(w, B=64)
    d = generate(small, "cpu")
    o, l = d["o"].numpy(), d["lse"].numpy()

    def unit(k):
        oracle.combine("f32", o[None], l[None], base=w.base, sanitize=True)
        return small.B / w.B

    el, done = run_oracle_units(unit, threads, budget_s)
    return el / done * 1e6, el, done


def time_oracle_peer_major(pm, budget_s: float, threads: int):
    """Oracle µs per call of a peer-major workload on `threads` host threads:
    share k is source k % N's interleaved pack and destination k % N's fused
    unpack+combine (1/N of a call each)."""
    import numpy as np

    import oracle

    w = pm["w"]
    o = host_payload(pm["d"]["o"])                  # [S, B, H, D]
    lse = pm["d"]["lse"].cpu().numpy()
    send = host_payload(pm["send"])                 # [S, N, B, H_pr, D + lpd]
    N, B, H_pr, D = w.N, w.B, w.H_pr, w.D
    lpd = 4 // pm["d"]["o"].element_size()

    def unit(k):
        s = k % N
        dst = np.empty((1, N, B, H_pr, D + lpd), dtype=o.dtype)
        oracle.pack(w.dtype, N, o[s:s + 1], lse[s:s + 1], dst[..., :D], dst.view(np.float32)[..., D // lpd])
        oracle.unpack_combine(w.dtype, send[None, :, s], D, base=w.base)  # destination s's rows
        return 1.0 / N

    el, done = run_oracle_units(unit, threads, budget_s)
    return el / done * 1e6, el, done


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def run_gpu(args):
    import torch

    from decode_context_attention_gb300 import binding, build

    rank, world = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if local == 0:
        build.build()
    barrier(device)
    binding.load()
    peak, peak_kind = load_peaks()
    cores = host_cores()
    flush = L2Flush(device)
    clocks = ClockSampler(local)
    clocks.start()

    if args.only:
        # a short run of one workload (for profiler captures); prints nothing
        wl = {"mla_decode": lambda: setup_mla_decode(device),
              "sweep": lambda: setup_sweep_max(device),
              "mla_decode_fp8": lambda: setup_mla_fp8(device),
              "decode_attention": lambda: setup_decode_attention(device, batch=args.att_batch),
              "gqa_decode_attention": lambda: setup_decode_attention(device, split_tokens=2048, batch=args.att_batch,
                                                                     name="gqa_decode_attention"),
              "two_collective": lambda: setup_two_collective(device),
              "per_rank": lambda: setup_per_rank(device),
              "cached_extend": lambda: setup_cached_extend(device, args.ext_tokens),
              "mla_decode_attention": lambda: setup_mla_attention(device, batch=args.att_batch)}[args.only]()
        time_sequence(wl["launches"], args.steps, args.warmup,
                      None if args.only == "cached_extend" else flush, device)
        clocks.stop()
        return

    # --- headline: MLA decode merge, pack + combine, all 8 ranks ----------------
    mla = setup_mla_decode(device, seed_offset=rank)
    per, wall = time_sequence(mla["launches"], args.steps, args.warmup, flush, device)
    step_ms = [sum(x) for x in zip(*per)]
    ms_per_step = max_over_ranks(statistics.fmean(step_ms), device)
    kernels = [kernel_record(n, p, b, peak) for n, p, b in zip(mla["names"], per, mla["bytes"])]
    # the pack's stores can still be in L2 at its end event: time it again with
    # their write-back to HBM inside the timed region
    wb_ms, evict_ms = time_with_writeback(mla["launches"][0], max(20, args.steps // 10), args.warmup, flush,
                                          device)
    pack_wb = kernel_record(mla["names"][0] + ", incl. the write-back of its L2-resident stores", [wb_ms],
                            mla["bytes"][0], peak)
    pack_wb["eviction_pass_us"] = round(evict_ms * 1e3, 3)
    kernels[0]["with_writeback"] = pack_wb

    # --- e2e: host buffers in, host result out, through the public binding ------
    e2e = None if args.no_e2e else run_e2e(mla, args, device)

    # --- secondary workloads (same run) ----------------------------------------
    secondary = []
    if not args.no_secondary:
        gm, gmed = time_graph_step(mla, max(50, args.steps // 4), args.warmup, flush, device)
        secondary.append({"workload": "mla_decode headline step captured as one CUDA graph (pack + combine), "
                                      "L2 flushed before each replay only",
                          "us_per_step": round(gm, 3), "us_median": round(gmed, 3),
                          "gpu_launches_per_step": 2})
        for setup, what in ((setup_per_rank, "per-rank calls (G=1) of the headline workload"),
                            (setup_two_collective, "two-collective layout: separate O and LSE buffers")):
            sw = setup(device)
            p2, _ = time_sequence(sw["launches"], max(20, args.steps // 10), args.warmup, flush, device)
            w2 = sw["w"]
            secondary.append({"workload": f"{w2.name} N={w2.N} B={w2.B} H={w2.H} D={w2.D} {w2.dtype} "
                                          f"base-{w2.base}, {what}",
                              "kernels": [kernel_record(n, p, b, peak)
                                          for n, p, b in zip(sw["names"], p2, sw["bytes"])]})
            del sw
        for setup in (setup_sweep_max, setup_mla_fp8):
            sw = setup(device)
            p2, _ = time_sequence(sw["launches"], max(20, args.steps // 10), args.warmup, flush, device)
            w2 = sw["w"]
            rec = {"workload": f"{w2.name} N={w2.N} B={w2.B} H={w2.H} D={w2.D} {w2.dtype} base-{w2.base}, "
                               "peer-major pack + fused unpack+combine",
                   "kernels": [kernel_record(n, p, b, peak)
                               for n, p, b in zip(sw["names"], p2, sw["bytes"])]}
            if rank == 0 and not args.no_cpu_baseline:
                us, el, n = time_oracle_peer_major(sw, min(5.0, args.cpu_budget), cores)
                rec["cpu_oracle"] = {"us_per_call": round(us, 1), "cores": cores,
                                     "sample": f"{n:.2f} calls as shares of one source's pack + one "
                                               f"destination's unpack+combine (1/{w2.N} of a call each), "
                                               f"{el:.1f} s on {cores} threads"}
            secondary.append(rec)
            del sw
        # splits of local tokens per CTA: 1024 for MHA, 2048 for GQA (measured
        # best among 256..2048: fewer split partials to write and merge)
        for att_name, att_split, att_page in (("mha_decode_attention", 1024, 0), ("gqa_decode_attention", 2048, 0),
                                              ("gqa_decode_attention", 2048, 64)):
            at = setup_decode_attention(device, split_tokens=att_split, name=att_name, page_size=att_page)
            p4, _ = time_sequence(at["launches"], max(10, args.steps // 20), 3, flush, device)
            rec = {"workload": f"{att_name}{f' over {att_page}-token pages' if att_page else ''} "
                               "(the step before the merge)",
                   "workspace_bytes": at["workspace_bytes"],
                   "kernels": [kernel_record(at["names"][0], p4[0], at["bytes"][0], peak)]}
            if rank == 0 and not args.no_cpu_baseline and not att_page:  # paging leaves the arithmetic alone
                us, el, n = time_oracle_attention(at, min(5.0, args.cpu_budget), cores)
                rec["cpu_oracle"] = {"us_per_call": round(us, 1), "cores": cores,
                                     "sample": f"sampled (request, head) rows worth {n:.2e} calls, {el:.1f} s "
                                               f"on {cores} threads, scaled by KV tokens"}
            secondary.append(rec)
            del at
            torch.cuda.empty_cache()
        mt = setup_mla_attention(device)
        p5, _ = time_sequence(mt["launches"], max(10, args.steps // 20), 3, flush, device)
        krec = kernel_record(mt["names"][0], p5[0], mt["bytes"][0], peak)
        tf = mt["flops"] / (statistics.fmean(p5[0]) * 1e-3) / 1e12
        tpeak, tkind = load_tensor_peak()
        krec.update({"flops": mt["flops"], "achieved_tflops": round(tf, 1), "tensor_peak_tflops": tpeak,
                     "frac_of_tensor_peak": round(tf / tpeak, 4), "tensor_peak_kind": tkind})
        rec = {"workload": "mla_decode_attention (absorbed MLA on the tcgen05 tensor cores; the step whose "
                           "outputs the MLA decode merge takes)",
               "workspace_bytes": mt["workspace_bytes"], "kernels": [krec]}
        if rank == 0 and not args.no_cpu_baseline:
            us, el, n = time_oracle_mla_attention(mt, min(5.0, args.cpu_budget), cores)
            rec["cpu_oracle"] = {"us_per_call": round(us, 1), "cores": cores,
                                 "sample": f"sampled (request, head) rows worth {n:.2e} calls, {el:.1f} s "
                                           f"on {cores} threads, scaled by latent rows"}
        secondary.append(rec)
        del mt
        torch.cuda.empty_cache()
        ce = setup_cached_extend(device, slices=True)
        p3, _ = time_sequence(ce["launches"], args.ext_steps, 3, None, device)
        rec = {"workload": "cached_extend N=8 T=16384 H=96 D=512 fp32",
               "inputs_vs_l2": "24 GiB stack, far larger than L2 (no flush)",
               "kernels": [kernel_record(n, p, b, peak) for n, p, b in zip(ce["names"], p3, ce["bytes"])]}
        if rank == 0 and not args.no_cpu_baseline:
            us, el, n = time_oracle_cached_extend(min(5.0, args.cpu_budget), cores)
            rec["cpu_oracle"] = {"us_per_call": round(us, 1), "cores": cores,
                                 "sample": f"all rows of the 64-token case, {n * 256:.0f} times, {el:.1f} s on "
                                           f"{cores} threads, scaled by rows"}
        secondary.append(rec)
        del ce
        torch.cuda.empty_cache()
    clk = clocks.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        us, el, n = time_oracle(mla, args.cpu_budget, cores)
        us1, el1, n1 = time_oracle(mla, min(5.0, args.cpu_budget), 1)
        cpu = {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n:.2f} calls as shares of one source's pack + one destination's combine "
                         f"(1/8 of a call each, every rank in turn), {el:.1f} s of fp64 C on {cores} "
                         "host threads",
               "single_core": {"value": round(us1, 1), "unit": UNIT, "cores": 1,
                               "sample": f"{n1:.2f} calls the same way, {el1:.1f} s on 1 thread"}}

    if rank != 0:
        return
    # the roofline names the combine: the kernel whose share of HBM peak the
    # merge is judged by (the pack, a bit copy, is reported beside it)
    k = kernels[1]
    traffic = ncu_traffic(mla["kernels"][1])
    w = mla["w"]
    line = {
        "metric": METRIC, "value": round(ms_per_step * 1e3, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded O ~ N(0,1), LSE ~ U(0,20) base 2)",
        "config": {"workload": f"mla_decode N={w.N} B={w.B} H={w.H} D={w.D} bf16 base-2, "
                               "peer-inside pack + combine over strided recv views, all ranks on "
                               "one GPU", "calls_per_step_per_gpu": 1,
                   "arithmetic": "bf16 payload and fp32 LSE; the pack is a bit copy, the merge "
                                 "accumulates in fp32 and rounds once to bf16",
                   "l2": "flushed before every kernel (2x-L2 write, then 2x-L2 read), outside "
                         "the timed events",
                   "parallelism": f"{world} independent replica(s), no collective"},
        "roofline": {"bound": "hbm", "kernel": k["kernel"], "achieved": k["achieved_gbs"],
                     "peak": peak, "unit": "GB/s", "frac": k["frac_of_measured_hbm"],
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "peak_theoretical_gbs": theoretical_hbm_gbs(local),
                     "traffic": traffic, "algorithmic_bytes": k["algorithmic_bytes"],
                     "duration_us": k["us_per_launch"],
                     "pack": {"kernel": kernels[0]["kernel"], "achieved": kernels[0]["achieved_gbs"],
                              "frac": kernels[0]["frac_of_measured_hbm"],
                              "traffic": ncu_traffic(mla["kernels"][0]),
                              "with_writeback": {"us": pack_wb["us_per_launch"],
                                                 "achieved": pack_wb["achieved_gbs"],
                                                 "frac": pack_wb["frac_of_measured_hbm"]},
                              "note": "a bit copy; its end event can fire while part of its stores "
                                      "are still in L2, so its time with their write-back "
                                      "included is given as well"}},
        "kernels": kernels,
        "secondary": secondary,
        "e2e": e2e,
        "gpu_launches": len(mla["launches"]) * args.steps,
        "cpu_baseline": cpu,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    print(json.dumps(line), flush=True)


def time_graph_step(mla, steps, warmup, flush, device):
    """The headline step (pack + combine) captured once as a CUDA graph and
    replayed; L2 is flushed before each replay only, so the combine may find
    the tail of the freshly written send buffer still in L2, as in a real
    back-to-back step.  Returns (mean, median) µs per step."""
    import torch

    from decode_context_attention_gb300 import binding, layouts

    d, w = mla["d"], mla["w"]
    dst_o, dst_lse = layouts.peer_inside_send_views(mla["partial_o"], mla["stats"])
    ro, rl = layouts.exchange_peer_inside(mla["partial_o"], mla["stats"])

    def step():
        binding.pack_send(d["o"], d["lse"], dst_o, dst_lse)
        binding.lse_combine(ro, rl, mla["out"], mla["out_lse"], base=w.base)

    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(device).wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    per, _ = time_sequence([g.replay], steps, warmup, flush, device)
    return statistics.fmean(per[0]) * 1e3, statistics.median(per[0]) * 1e3


def run_e2e(mla, args, device, chunks=4):
    """µs per call with the inputs in pinned host memory and the result
    written to pinned host memory, all inside the timed region.  The pack reads
    the host inputs directly over the host link (the upload is fused into it)
    and the combine writes the merged rows and LSEs straight to host memory.
    The tokens are taken in `chunks` slices: the pack of slice c+1 (host ->
    device traffic) runs on one stream while the combine of slice c (device ->
    host traffic) runs on another, so the two directions of the link overlap;
    each call ends with both streams joined."""
    import torch

    from decode_context_attention_gb300 import binding, layouts

    d, w = mla["d"], mla["w"]
    o_h = d["o"].cpu().pin_memory()
    l_h = d["lse"].cpu().pin_memory()
    out_h = torch.empty(mla["out"].shape, dtype=mla["out"].dtype).pin_memory()
    lse_h = torch.empty(mla["out_lse"].shape, dtype=torch.float32).pin_memory()
    dst_o, dst_lse = layouts.peer_inside_send_views(mla["partial_o"], mla["stats"])
    ro, rl = layouts.exchange_peer_inside(mla["partial_o"], mla["stats"])
    B = o_h.shape[1]
    bounds = [(B * c // chunks, B * (c + 1) // chunks) for c in range(chunks)]
    sp, sc = torch.cuda.Stream(device), torch.cuda.Stream(device)
    packs = [binding.prepare_pack_send(o_h[:, b0:b1], l_h[:, b0:b1], dst_o[:, :, b0:b1], dst_lse[:, :, b0:b1],
                                       stream=sp) for b0, b1 in bounds]
    combs = [binding.prepare_lse_combine(ro[:, :, b0:b1], rl[:, :, b0:b1], out_h[:, b0:b1], lse_h[:, b0:b1],
                                         base=w.base, stream=sc) for b0, b1 in bounds]
    ready = [torch.cuda.Event() for _ in bounds]

    def step():
        for c in range(chunks):
            packs[c]()
            ready[c].record(sp)
            sc.wait_event(ready[c])
            combs[c]()
        sp.wait_stream(sc)

    steps = max(10, args.steps // 20)
    sp.wait_stream(torch.cuda.current_stream(device))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    barrier(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(sp)
    for _ in range(steps):
        step()
    b.record(sp)
    torch.cuda.synchronize(device)
    ms = max_over_ranks(a.elapsed_time(b) / steps, device)
    # the host result is the device path's, bit for bit
    mla["launches"][0]()
    mla["launches"][1]()
    torch.cuda.synchronize(device)
    if not (torch.equal(out_h.view(torch.int16), mla["out"].cpu().view(torch.int16))
            and torch.equal(lse_h, mla["out_lse"].cpu())):
        raise RuntimeError("host-buffer path differs from the device path")
    h2d = o_h.numel() * o_h.element_size() + l_h.numel() * 4
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4
    return {"value": round(ms * 1e3, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "api": "decode_context_attention_gb300.binding.pack_send + lse_combine on pinned host "
                   "tensors (inputs read and result written over the host link)",
            "pipeline": f"{chunks} token slices; pack (host->device reads) on one stream, combine "
                        "(device->host writes) on another, joined at the end of each call"}


def run_reference(args):
    """The fp64 CPU oracle on a bounded sample of the same workload, same unit."""
    import torch

    rank, world = dist_env()[0], dist_env()[1]
    if world > 1 and rank != 0:
        return
    from decode_context_attention_gb300.workloads import WORKLOADS, generate

    w = WORKLOADS["mla_decode"]
    d = generate(w, "cpu")
    S, B, H, D = d["o"].shape
    partial_o = d["o"].view(S, B, w.N, w.H_pr, D).permute(0, 1, 3, 2, 4).contiguous()
    stats = torch.zeros((S, B, w.H_pr, w.N, 2))
    stats[..., 0] = d["lse"].view(S, B, w.N, w.H_pr).permute(0, 1, 3, 2)
    mla = {"d": d, "w": w, "partial_o": partial_o, "stats": stats}
    inputs = oracle_host_inputs(mla)
    cores = host_cores()
    # one step: every source's pack and every destination's combine over the
    # first `rows` tokens, split into at least `cores` independent shares
    # (rank x token range) run on `cores` host threads
    chunks = max(1, -(-cores // w.N))

    def tasks(rows):
        cuts = [rows * c // chunks for c in range(chunks + 1)]
        return [(k, cuts[c], cuts[c + 1]) for k in range(w.N) for c in range(chunks) if cuts[c + 1] > cuts[c]]

    def step(rows, pool):
        return sum(pool.map(lambda t: oracle_mla_unit(inputs, *t), tasks(rows)))

    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(max_workers=cores) as pool:
        # size each step so warmup + steps finish in about two minutes
        t0 = time.perf_counter()
        step(min(B, 2 * chunks), pool)
        per_row = (time.perf_counter() - t0) / min(B, 2 * chunks)
        budget = 120.0 / max(1, args.steps + args.warmup + 2)
        rows = int(max(1, min(B, budget / max(per_row, 1e-9))))
        for _ in range(args.warmup):
            step(rows, pool)
        times = []
        frac = None
        for _ in range(args.steps):
            t = time.perf_counter()
            frac = step(rows, pool)
            times.append(time.perf_counter() - t)
    us = statistics.fmean(times) / frac * 1e6
    # the same shares one after the other on one thread, once
    t = time.perf_counter()
    frac1 = sum(oracle_mla_unit(inputs, *tk) for tk in tasks(rows))
    us1 = (time.perf_counter() - t) / frac1 * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": {"workload": f"mla_decode N={w.N} B={w.B} H={w.H} D={w.D} bf16 base-2, "
                               "peer-inside pack + combine"},
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: every source's pack + every destination's combine "
                                   f"over the first {rows} of {B} tokens, as {len(tasks(rows))} shares "
                                   f"on {cores} host threads, scaled to one call",
                         "single_core": {"value": round(us1, 1), "unit": UNIT, "cores": 1,
                                         "sample": "the same shares one after the other on 1 thread, once"}},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--ext-steps", type=int, default=40, help="timed calls of the 29 GB workload")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["mla_decode", "sweep", "mla_decode_fp8", "two_collective", "per_rank",
                                       "cached_extend", "decode_attention", "gqa_decode_attention",
                                       "mla_decode_attention"],
                    help="run just this workload's launches (profiling); no JSON line")
    ap.add_argument("--att-batch", type=int, default=None,
                    help="requests of the decode-attention workload under --only (default 64)")
    ap.add_argument("--ext-tokens", type=int, default=None,
                    help="tokens of the cached-extend workload under --only (default 16384)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
