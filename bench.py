"""Benchmark: paged decode over a 2-GiB-per-pool paged K/V cache on GB300.

Default workload: Llama-3-8B-shaped bf16 decode (B=256, one query token,
Hq=32, Hkv=8, D=128, 4096 keys per sequence, page_size 16, 65536 shuffled pages
per pool = 2 GiB each).  A step is one pass of the whole hot path over the
batch: the paged forward (block-table gather, staging, QK, mask, online
softmax, PV, per-split finalise) and, when split_kv > 1, the combine.

Prints one JSON line.  ``value`` is algorithmic bytes per step / step time
(GB/s), where algorithmic bytes = the K and V bytes of every valid token + q +
out + the block-table ids read; inputs (2 x 2 GiB) exceed L2, so no flush is
needed between steps.  ``--impl reference`` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "paged decode KV-read HBM GB/s and % of GB300 peak; µs per decode step"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=250)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_decode",
                    choices=["llama8b_decode", "over2gib_decode", "ragged_decode", "causal_prefill", "tiny_decode_f32",
                             "llama8b_decode_fp8", "llama8b_decode_int8", "mixed_decode_prefill", "d256_decode",
                             "mha_decode", "causal_prefill_f16", "llama8b_decode_over2gib"])
    ap.add_argument("--split-kv", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences (llama8b/over2gib workloads only; smaller pools for profiling)")
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="variable-length batches: the plain call (its two kernels one after the other)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="the Llama-3-8B decode line without its over-2-GiB and prefill keys")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = os.environ.get("PA_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    """Slowest rank's value (step times are taken as the max over ranks)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: int, ws: int, ms_step: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return bytes_per_rank_step * ws / (ms_step * 1e-3) / 1e9


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, max clock, throttle reasons)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled=True):
        self.index, self.enabled, self.lines, self.proc = index, enabled, [], None

    def __enter__(self):
        if self.enabled:
            try:
                self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                              "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
                self.thread = threading.Thread(target=self._read, daemon=True)
                self.thread.start()
                time.sleep(0.3)
            except OSError:
                self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                return json.load(f)
        except (OSError, ValueError):
            return None
    return None


def algorithmic_bytes(wl, split_kv: int) -> dict:
    """Bytes a decode step must move: valid K and V tokens, q, out, block-table ids, seq_lens, and
    for quantized pools the K and V scale of every (page read, kv head)."""
    L = wl.seq_lens.astype(np.int64)
    kv = int(L.sum()) * wl.Hkv * wl.D * wl.kv_esize * 2
    q = wl.B * wl.Sq * wl.Hq * wl.D * wl.esize
    out = q
    ids = int(wl.nblk().sum()) * 4 + wl.B * 4
    scales = int(wl.nblk().sum()) * wl.Hkv * 4 * 2 if wl.kv_dtype is not None else 0
    return {"kv": kv, "q": q, "out": out, "ids": ids, "scales": scales, "total": kv + q + out + ids + scales}


def causal_flops(wl) -> float:
    """Useful flops of a step: 4*D per (query row, valid key) pair (QK^T and PV), masked work excluded."""
    L = wl.seq_lens.astype(np.int64)
    pairs = 0
    for b in range(wl.B):
        if wl.causal:
            qoff = int(L[b]) - wl.Sq if wl.q_offset is None else int(wl.q_offset[b])
            reach = np.clip(qoff + np.arange(wl.Sq) + 1, 0, int(L[b]))
            pairs += int(reach.sum())
        else:
            pairs += int(L[b]) * wl.Sq
    return 4.0 * wl.D * pairs * wl.Hq


KERNEL_SOURCES = {
    "paged_attn_mma_kernel": ("attn_mma.cu", "mma_common.cuh", "common.cuh", "kernels.h"),
    "paged_attn_kvq_decode_kernel": ("attn_mma_kvq.cu", "mma_common.cuh", "common.cuh", "kernels.h"),
    "paged_attn_kvq_prefill_kernel": ("attn_mma_kvq.cu", "mma_common.cuh", "common.cuh", "kernels.h"),
    # the variable-length call: the tcgen05 kernel (long sequences) and the one-grid kernel
    "paged_attn_mma_varlen_kernel": ("attn_mma.cu", "mma_common.cuh", "attn_tc05.cu", "tc05.cuh", "common.cuh",
                                     "kernels.h"),
    "paged_attn_mma_t_kernel": ("attn_mma_t.cu", "mma_common.cuh", "common.cuh", "kernels.h"),
    "paged_attn_tc05_kernel": ("attn_tc05.cu", "tc05.cuh", "common.cuh", "kernels.h"),
    "paged_attn_simt_kernel": ("attn_simt.cu", "common.cuh", "kernels.h"),
    "paged_attn_simt_decode_kernel": ("attn_simt_decode.cu", "mma_common.cuh", "common.cuh", "kernels.h"),
}


def kernel_source_digest(kernel: str) -> str:
    """Hash of the sources a kernel is built from (a recorded ncu traffic figure is only valid for it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_201_gb300", "csrc")
    for name in KERNEL_SOURCES.get(kernel, ()):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, split_kv: int):
    """DRAM bytes per launch from a committed ncu summary of this kernel, workload and split_kv, if it
    was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(f"{kernel}/{workload}/split{split_kv}")
    if not ent or ent.get("source_digest") != kernel_source_digest(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def traffic_fields(kernel: str, workload: str, split_kv: int) -> dict:
    """``traffic`` and where it comes from: the bench does not run ncu, so the figure is one recorded
    by an ncu capture of the same kernel, workload and split (profiles/traffic.json), valid only for
    the kernel sources it was taken on (their digest); null when those sources have changed since."""
    t = recorded_traffic(kernel, workload, split_kv)
    return {"traffic": t,
            "traffic_source": None if t is None else (
                f"recorded: ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                f"profiles/traffic.json entry {kernel}/{workload}/split{split_kv}, "
                f"kernel source digest {kernel_source_digest(kernel)}")}


def build_workload(name, batch=None):
    from paged_kv_cache_201_gb300 import workloads as W
    if batch is not None and name in ("llama8b_decode", "over2gib_decode", "llama8b_decode_fp8", "llama8b_decode_over2gib",
                                      "llama8b_decode_int8", "d256_decode", "mha_decode"):
        return W.make(name, B=batch)
    return W.make(name)


def cpu_sample_rows(wl, n_seq: int):
    """Rows (b, i, h) of the first n_seq sequences, every query token and head."""
    import oracle
    rows = oracle.all_rows(n_seq, wl.Sq, wl.Hq)
    return rows


def time_oracle(wl, k_host, v_host, split_kv: int, n_seq: int, scales=None):
    """Run the oracle on the first n_seq sequences; return (seconds, kv_bytes_processed, threads).
    ``scales`` = (k_scale, v_scale) host arrays for quantized pools."""
    import oracle
    rows = cpu_sample_rows(wl, n_seq)
    t0 = time.perf_counter()
    if wl.kv_dtype is not None:
        oracle.workload_rows_kvq(wl, split_kv=split_kv, row_bih=rows, k_cache=k_host, v_cache=v_host,
                                 k_scale=scales[0], v_scale=scales[1], want_split=split_kv > 1)
    else:
        oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows, k_cache=k_host, v_cache=v_host,
                             want_split=split_kv > 1)
    dt = time.perf_counter() - t0
    kv = int(wl.seq_lens[:n_seq].astype(np.int64).sum()) * wl.Hkv * wl.D * wl.kv_esize * 2
    return dt, kv, oracle.num_threads()


def host_pools(wl, k, v):
    """Device pools -> host element arrays for the oracle (uint16 bits, float32, or uint8 bits of
    8-bit elements)."""
    import torch
    if wl.kv_dtype is not None:
        return k.cpu().numpy(), v.cpu().numpy()
    if wl.dtype == "f32":
        return k.cpu().numpy(), v.cpu().numpy()
    return k.view(torch.int16).cpu().numpy().view(np.uint16), v.view(torch.int16).cpu().numpy().view(np.uint16)


def data_text(wl) -> str:
    if wl.kv_dtype == "fp8e4m3":
        return ("synthetic (seeded N(0,1) K/V quantized to FP8 E4M3 with per-(page, kv head) scales "
                "max|x|/448; N(0,1) q rounded to bf16; shuffled pages)")
    if wl.kv_dtype == "int8":
        return ("synthetic (seeded N(0,1) K/V quantized to int8 with per-(page, kv head) scales "
                "max|x|/127, round to nearest even; N(0,1) q rounded to bf16; shuffled pages)")
    return f"synthetic (seeded N(0,1) rounded to {wl.dtype}; shuffled pages)"


L2_BYTES = 129 * 2 ** 20


def pool_bytes(wl) -> int:
    return wl.num_pages * wl.page_size * wl.Hkv * wl.D * wl.kv_esize


def l2_text(wl) -> str:
    pool = pool_bytes(wl)
    if 2 * pool > L2_BYTES:
        return f"inputs (2 x {pool / 2 ** 30:.2f} GiB pools) larger than L2"
    return (f"inputs (2 x {pool / 2 ** 20:.1f} MiB pools) smaller than L2: a 256 MiB buffer is written before "
            "each timed step, outside its events")


# ----------------------------------------------------------------------------- timing protocol
N_BATCHES = 5


def batch_sizes(K: int, n: int = N_BATCHES):
    """K timed steps cut into n batches as equal as possible (fewer batches when K < n)."""
    n = max(1, min(n, K))
    return [K // n + (1 if j < K % n else 0) for j in range(n)]


def timed_batches(fns, K: int, stream, flush=None):
    """The timing protocol of rocm-libraries PR #14349 (Performance): after the caller's warm-up, the
    K timed steps run as N_BATCHES batches, each bracketed by CUDA events on the launching stream; a
    step's time is the median over batches of (batch time / steps in the batch).

    ``fns`` is a list of callables that together make one step; the events around the first one
    also give its own median time (the forward kernel when the second is the combine).  With
    ``flush`` (a device buffer larger than L2) the buffer is written before every step and the
    step's time is the sum of its own events, so the flush is not counted.
    Returns (ms per step, ms of fns[0] per step)."""
    import torch
    sizes = batch_sizes(K)
    step_ms, first_ms = [], []
    for j, n in enumerate(sizes):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for i in range(n):
            if flush is not None:
                flush.fill_((j * 131 + i) & 0xFF)
            ev[i][0].record(stream)
            fns[0]()
            ev[i][1].record(stream)
            for f in fns[1:]:
                f()
            ev[i][2].record(stream)
        b1.record(stream)
        torch.cuda.synchronize()
        first_ms.append(sum(e[0].elapsed_time(e[1]) for e in ev) / n)
        if flush is not None:
            step_ms.append(sum(e[0].elapsed_time(e[2]) for e in ev) / n)
        else:
            step_ms.append(b0.elapsed_time(b1) / n)
    return float(np.median(step_ms)), float(np.median(first_ms))


E2E_TIMING = ("value / ms_per_step: host wall clock (time.perf_counter) from a synchronised device to the "
              "synchronize after the batch's last read-back, median of 5 batches, so host launch and copy-issue "
              "costs count; event_value / event_ms_per_step: CUDA events from the batch's first upload to its "
              "last read-back")
E2E_PIPELINING = ("every step uploads its inputs from pinned host memory, makes the public call and reads its "
                  "outputs back to pinned host memory; two buffer sets let step i+1's upload and step i-1's "
                  "read-back run on copy streams while step i computes, as a serving loop does")


class PipelinedE2E:
    """End-to-end steps the way a serving loop runs them: every step uploads its inputs from pinned
    host memory, makes the public call and reads its results back to pinned host memory, with two
    buffer sets so that step i + 1's upload and step i - 1's read-back run on copy streams while step
    i computes.  Each step's own copies are in the timed region; events order every reuse of a buffer
    (an upload waits until the call two steps earlier has read that set, a call until the read-back
    two steps earlier has left its outputs).

    host_in: pinned host tensors; dev_in(j): device tensors of set j in the same order; dev_out(j) /
    host_out(j): the call's outputs and their pinned host copies; call(ins, outs, stream) runs one
    step on `stream`."""

    def __init__(self, host_in, dev_in, dev_out, host_out, call, stream):
        import torch
        self.torch, self.host_in, self.call, self.stream = torch, host_in, call, stream
        self.dev_in = [dev_in(j) for j in range(2)]
        self.dev_out = [dev_out(j) for j in range(2)]
        self.host_out = [host_out(j) for j in range(2)]
        self.h2d, self.d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.in_ready, self.in_free, self.out_ready, self.out_free = ev(), ev(), ev(), ev()
        self.i = 0

    def step(self):
        torch = self.torch
        j, first = self.i & 1, self.i < 2
        with torch.cuda.stream(self.h2d):
            if not first:
                self.h2d.wait_event(self.in_free[j])
            for dst, src in zip(self.dev_in[j], self.host_in):
                dst.copy_(src, non_blocking=True)
            self.in_ready[j].record(self.h2d)
        self.stream.wait_event(self.in_ready[j])
        if not first:
            self.stream.wait_event(self.out_free[j])
        self.call(self.dev_in[j], self.dev_out[j], self.stream)
        self.in_free[j].record(self.stream)
        self.out_ready[j].record(self.stream)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.out_ready[j])
            for dst, src in zip(self.host_out[j], self.dev_out[j]):
                dst.copy_(src, non_blocking=True)
            self.out_free[j].record(self.d2h)
        self.i += 1

    def bytes(self):
        h = sum(t.numel() * t.element_size() for t in self.host_in)
        d = sum(t.numel() * t.element_size() for t in self.host_out[0])
        return int(h), int(d)


def e2e_pipelined_batches(pipe, K: int):
    """K pipelined steps in N_BATCHES batches, each from a synchronised device to a synchronize after
    its last read-back.  Returns (median event ms per step, first upload to last read-back; median
    host wall-clock ms per step)."""
    import torch
    ev_ms, wall_ms = [], []
    for n in batch_sizes(K):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        a.record(pipe.h2d)
        for _ in range(n):
            pipe.step()
        b.record(pipe.d2h)
        torch.cuda.synchronize()
        wall_ms.append((time.perf_counter() - t0) * 1e3 / n)
        ev_ms.append(a.elapsed_time(b) / n)
    return float(np.median(ev_ms)), float(np.median(wall_ms))


# ----------------------------------------------------------------------------- further workloads in the headline line
def prepare_16bit(wl, S: int, dev, stream, variant: int = 0):
    """Device tensors of a 16-bit-pool workload and the callables of one step: the forward and, for
    S > 1, the combine."""
    import torch
    import paged_kv_cache_201_gb300 as pa
    from paged_kv_cache_201_gb300 import workloads as W
    t = {"q": W.host_to_torch(wl.q, wl.dtype).to(dev)}
    if wl.k_cache is not None:
        t["k"], t["v"] = W.host_to_torch(wl.k_cache, wl.dtype).to(dev), W.host_to_torch(wl.v_cache, wl.dtype).to(dev)
    else:
        t["k"], t["v"] = W.fill_device_cache(wl, dev)
    t["bt"] = torch.from_numpy(wl.block_table).to(dev)
    t["sl"] = torch.from_numpy(wl.seq_lens).to(dev)
    t["qo"] = None if wl.q_offset is None else torch.from_numpy(wl.q_offset).to(dev)
    B, Sq, Hq, D = wl.B, wl.Sq, wl.Hq, wl.D
    t["out"] = torch.empty_like(t["q"])
    t["lse"] = torch.empty((B, Sq, Hq), dtype=torch.float32, device=dev)
    if S > 1:
        t["po"] = torch.empty((S, B, Sq, Hq, D), dtype=torch.float32, device=dev)
        t["pl"] = torch.empty((S, B, Sq, Hq), dtype=torch.float32, device=dev)
    o, l = (t["out"], t["lse"]) if S == 1 else (t["po"], t["pl"])

    def fwd():
        pa.paged_attn_fwd_variant(t["q"], t["k"], t["v"], t["bt"], t["sl"], wl.causal, t["qo"], S, wl.scale, o, l,
                                  variant, stream)

    fns = [fwd]
    if S > 1:
        fns.append(lambda: pa.paged_attn_combine(t["po"], t["pl"], t["out"], t["lse"], stream))
    return t, fns


def warm(fns, n):
    import torch
    for _ in range(max(n, 3)):
        for f in fns:
            f()
    torch.cuda.synchronize()


def interleaved_batches(fns_a, fns_b, K: int, stream):
    """Two workloads timed in alternating batches (a, b, a, b, ...; N_BATCHES each of the K-step
    protocol), so that both see the same clocks and the same state of the GPU.  Returns the two
    median ms per step."""
    import torch
    ms_a, ms_b = [], []
    for n in batch_sizes(K):
        for fns, acc in ((fns_a, ms_a), (fns_b, ms_b)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                for f in fns:
                    f()
            e1.record(stream)
            torch.cuda.synchronize()
            acc.append(e0.elapsed_time(e1) / n)
    return float(np.median(ms_a)), float(np.median(ms_b))


def extra_workloads(args, dev, stream, headline_fns, headline_bytes, hbm_peak, tensor_peak):
    """The other targets of the headline in the same run and on the same GPU:
    - ``over2gib``: the over-2^31-byte decode (B=256, Hq=64, Hkv=4, L=8192, 135168 pages per pool,
      split 4), every sequence reading pages on both sides of byte 2^31;
    - ``over2gib_same_shape``: the headline's own shape over pools of 65536 + 2048 pages, every
      sequence holding pages on both sides of byte 2^31, timed in batches alternating with the
      headline workload; ``ratio`` is its GB/s over the headline's (1.0 = no slowdown past 2^31);
    - ``prefill``: the causal prefill (B=4, Sq=1024, GQA 32/8, q_offset up to 3072) at split 8 and 1,
      useful (causal) flops per second against the measured bf16 burst peak.
    Each runs the K-step protocol of the headline (warm-up, N_BATCHES batches, median)."""
    import torch
    from paged_kv_cache_201_gb300 import workloads as W
    K = args.steps
    res = {}

    wl = W.llama8b_decode_over2gib()
    t, fns = prepare_16bit(wl, 1, dev, stream)
    warm(fns, args.warmup)
    warm(headline_fns, 2)
    ms_ref, ms_hi = interleaved_batches(headline_fns, fns, K, stream)
    ab = algorithmic_bytes(wl, 1)
    assert ab["total"] == headline_bytes
    res["over2gib_same_shape"] = {
        "workload": "llama8b_decode_over2gib", "num_pages": wl.num_pages, "split_kv": 1,
        "pool_bytes": pool_bytes(wl), "pages_past_2gib_per_sequence": int(
            (wl.block_table >= W.LLAMA_OVER2G_FIRST_HIGH).sum(axis=1).min()),
        "us_per_step": round(ms_hi * 1e3, 2), "value": round(ab["total"] / (ms_hi * 1e-3) / 1e9, 1),
        "headline_us_per_step": round(ms_ref * 1e3, 2),
        "headline_value": round(headline_bytes / (ms_ref * 1e-3) / 1e9, 1),
        "ratio": round(ms_ref / ms_hi, 4), "unit": "GB/s",
        "how": "alternating batches with the headline workload (65536-page pools, below 2^31 bytes)"}
    del t, fns
    torch.cuda.empty_cache()

    wl = W.over2gib_decode()
    t, fns = prepare_16bit(wl, 4, dev, stream)
    warm(fns, args.warmup)
    ms, fwd_ms = timed_batches(fns, K, stream)
    ab = algorithmic_bytes(wl, 4)
    res["over2gib"] = {
        "workload": "over2gib_decode", "num_pages": wl.num_pages, "pool_bytes": pool_bytes(wl), "split_kv": 4,
        "us_per_step": round(ms * 1e3, 2), "value": round(ab["total"] / (ms * 1e-3) / 1e9, 1),
        "frac": round(ab["total"] / (ms * 1e-3) / 1e9 / hbm_peak, 4),
        "kernel": "paged_attn_mma_kernel", "kernel_us": round(fwd_ms * 1e3, 2),
        "kernel_frac": round(ab["total"] / (fwd_ms * 1e-3) / 1e9 / hbm_peak, 4), "unit": "GB/s",
        "bytes_per_step": ab["total"], **traffic_fields("paged_attn_mma_kernel", "over2gib_decode", 4)}
    del t, fns
    torch.cuda.empty_cache()

    wl = W.causal_prefill()
    fl = causal_flops(wl)
    pre = {"workload": "causal_prefill", "flops_per_step": fl, "unit": "TFLOP/s", "peak": tensor_peak,
           "kernel": "paged_attn_tc05_kernel"}
    for S in (8, 1):
        t, fns = prepare_16bit(wl, S, dev, stream)
        warm(fns, args.warmup)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # inputs (2 x 32 MiB pools) fit in L2
        ms, fwd_ms = timed_batches(fns, K, stream, flush)
        pre[f"split{S}"] = {
            "us_per_step": round(ms * 1e3, 2), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
            "frac": round(fl / (ms * 1e-3) / 1e12 / tensor_peak, 4), "kernel_us": round(fwd_ms * 1e3, 2),
            "kernel_tflops": round(fl / (fwd_ms * 1e-3) / 1e12, 1),
            "kernel_frac": round(fl / (fwd_ms * 1e-3) / 1e12 / tensor_peak, 4),
            **traffic_fields("paged_attn_tc05_kernel", "causal_prefill", S)}
        del t, fns, flush
    pre["l2"] = "pools smaller than L2: a 256 MiB buffer is written before each step, outside its events"
    res["prefill"] = pre
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- our arm
def run_ours(args, ws, rank, local):
    import torch
    import paged_kv_cache_201_gb300 as pa
    from paged_kv_cache_201_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load_library()
    wl = build_workload(args.workload, args.batch)
    S = args.split_kv or wl.split_kv[0]
    q = W.host_to_torch(wl.q, wl.dtype).to(dev)
    kvq = wl.kv_dtype is not None
    kv_code = {"fp8e4m3": pa.PA_FP8_E4M3, "int8": pa.PA_INT8}.get(wl.kv_dtype)
    ks = vs = None
    if kvq:
        if wl.k_cache is not None:
            k, v = torch.from_numpy(wl.k_cache).to(dev), torch.from_numpy(wl.v_cache).to(dev)
            ks, vs = torch.from_numpy(wl.k_scale).to(dev), torch.from_numpy(wl.v_scale).to(dev)
        else:
            k, v, ks, vs = W.fill_device_cache_q8(wl, dev)
    elif wl.k_cache is not None:
        k = W.host_to_torch(wl.k_cache, wl.dtype).to(dev)
        v = W.host_to_torch(wl.v_cache, wl.dtype).to(dev)
    else:
        k, v = W.fill_device_cache(wl, dev)
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    qo = None if wl.q_offset is None else torch.from_numpy(wl.q_offset).to(dev)
    B, Sq, Hq, D = wl.B, wl.Sq, wl.Hq, wl.D
    out = torch.empty_like(q)
    lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=dev)
    po = torch.empty((S, B, Sq, Hq, D), dtype=torch.float32, device=dev) if S > 1 else None
    pl = torch.empty((S, B, Sq, Hq), dtype=torch.float32, device=dev) if S > 1 else None
    stream = torch.cuda.current_stream(dev)

    def fwd():
        o, l = (out, lse) if S == 1 else (po, pl)
        if kvq:
            pa.paged_attn_fwd_kvq(q, k, v, ks, vs, bt, sl, wl.causal, qo, S, wl.scale, o, l, stream, kv_code)
        else:
            pa.paged_attn_fwd_variant(q, k, v, bt, sl, wl.causal, qo, S, wl.scale, o, l, args.variant, stream)

    def step():
        fwd()
        if S > 1:
            pa.paged_attn_combine(po, pl, out, lse, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    K = args.steps
    # Inputs smaller than L2 would stay resident between steps: then a 256 MiB buffer is written
    # before every step, outside the step's events, and the step time is the sum of those events.
    flush = pool_bytes(wl) * 2 <= L2_BYTES
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    fns = [fwd] + ([lambda: pa.paged_attn_combine(po, pl, out, lse, stream)] if S > 1 else [])
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        ms_local, fwd_ms = timed_batches(fns, K, stream, flush_buf)
    barrier(ws)
    ms_step = max_over_ranks(ms_local, ws, dev)
    flags = pa.paged_attn_last_error_word()
    if flags:
        raise RuntimeError(f"device error word {flags:#x} during the bench")

    ab = algorithmic_bytes(wl, S)
    value = job_throughput(ab["total"], ws, ms_step)
    hot = None
    if flush and ws == 1:
        # Pools that fit in L2 are reported cold (above: the flush before every step) and hot: the
        # same steps back to back, the pools resident in L2 after the first.
        hot_ms, _ = timed_batches(fns, K, stream, None)
        hot = {"ms_per_step": round(hot_ms, 5), "us_per_step": round(hot_ms * 1e3, 2),
               "value": round(job_throughput(ab["total"], 1, hot_ms), 1), "unit": "GB/s",
               "how": "the same steps and protocol with no L2 flush between steps (the pools stay resident)"}
    peaks = measured_peaks()
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    prefill = wl.Sq * wl.G > 16
    if kvq:
        kname = "paged_attn_kvq_prefill_kernel" if wl.Sq * wl.G > 16 else "paged_attn_kvq_decode_kernel"
    elif wl.D == 256 and wl.dtype != "f32" and wl.Sq * wl.G > 1 and args.variant in (0, 5):
        kname = "paged_attn_mma_t_kernel"
    elif wl.Sq * wl.G == 1 and wl.dtype != "f32" and wl.D != 256 and args.variant in (0, 1):
        kname = "paged_attn_simt_decode_kernel"
    elif args.variant:
        kname = {1: "paged_attn_simt_kernel", 4: "paged_attn_tc05_kernel"}.get(args.variant, "paged_attn_mma_kernel")
    else:  # what the planner picks for this shape
        kname = "paged_attn_tc05_kernel" if (prefill and wl.Sq * wl.G >= 64 and wl.D == 128 and 128 % wl.G == 0
                                             and wl.dtype != "f32") else (
            "paged_attn_simt_kernel" if (wl.dtype == "f32" or wl.Sq * wl.G <= 1) else "paged_attn_mma_kernel")
    fwd_bytes = ab["total"]
    achieved = fwd_bytes / (fwd_ms * 1e-3) / 1e9

    if prefill:
        # causal prefill is a dense contraction: the tensor pipe bounds it (useful flops only)
        tf_achieved = causal_flops(wl) / (fwd_ms * 1e-3) / 1e12
        if peaks and peaks.get("bf16_tflops"):
            tpeak, tpeak_src = float(peaks["bf16_tflops"]), "measured"
        else:
            tpeak, tpeak_src = FALLBACK_BF16_TFLOPS, "fallback"
        roofline = {"bound": "tensor", "kernel": kname, "achieved": round(tf_achieved, 1), "peak": tpeak,
                    "peak_source": tpeak_src, "unit": "TFLOP/s", "frac": round(tf_achieved / tpeak, 4),
                    "kernel_ms": round(fwd_ms, 5), **traffic_fields(kname, args.workload, S)}
    else:
        roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
                    "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "kernel_ms": round(fwd_ms, 5), **traffic_fields(kname, args.workload, S)}

    extras = {}
    if args.workload == "llama8b_decode" and ws == 1 and S == 1 and args.variant == 0 and not args.no_extras:
        tpeak_x = float(peaks["bf16_tflops"]) if peaks and peaks.get("bf16_tflops") else FALLBACK_BF16_TFLOPS
        extras = extra_workloads(args, dev, stream, fns, ab["total"], peak, tpeak_x)

    # ---- end to end through the public API: host inputs in, host result out, every step
    e2e = None
    if not args.no_e2e:
        host_in = [q.cpu().pin_memory(), bt.cpu().pin_memory(), sl.cpu().pin_memory()]
        wsp_bytes = pa.paged_attn_workspace_bytes(q, k, bt, S)
        wsp = torch.empty(max(wsp_bytes, 256), dtype=torch.uint8, device=dev)

        def call(ins, outs, st):
            # the single public call: split forward into the workspace, then the combine
            qd, btd, sld = ins
            od, ld = outs
            if kvq:
                pa.paged_attn_fwd_kvq_splitkv(qd, k, v, ks, vs, btd, sld, wl.causal, qo, S, wl.scale, od, ld, wsp,
                                              stream=st, kv_dtype=kv_code)
            else:
                pa.paged_attn_fwd_splitkv(qd, k, v, btd, sld, wl.causal, qo, S, wl.scale, od, ld, wsp, stream=st)

        pipe = PipelinedE2E(host_in, lambda j: [torch.empty_like(t, device=dev) for t in host_in],
                            lambda j: [torch.empty_like(out), torch.empty_like(lse)],
                            lambda j: [torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                                       torch.empty(lse.shape, dtype=lse.dtype).pin_memory()], call, stream)
        for _ in range(3):
            pipe.step()
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ev_ms, e2e_wall_ms = e2e_pipelined_batches(pipe, max(10, K // 4))
        e2e_ms = max_over_ranks(e2e_wall_ms, ws, dev)
        e2e_ev_ms = max_over_ranks(e2e_ev_ms, ws, dev)
        hb, db = pipe.bytes()
        e2e = {"value": round(job_throughput(ab["total"], ws, e2e_ms), 1), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db,
               "timing": E2E_TIMING, "pipelining": E2E_PIPELINING,
               "event_value": round(job_throughput(ab["total"], ws, e2e_ev_ms), 1),
               "event_ms_per_step": round(e2e_ev_ms, 4),
               "api": ("paged_attn_fwd_kvq_splitkv" if kvq else "paged_attn_fwd_splitkv") +
                      " (host q / block table / seq_lens in, host out / lse back)"}

    # ---- CPU baseline: the oracle on a bounded sample of the same workload (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        k_h, v_h = host_pools(wl, k, v)
        sc_h = (ks.cpu().numpy(), vs.cpu().numpy()) if kvq else None
        # one pass over the whole batch calibrates; then whole-batch passes until >= 10 s (cap 30 s)
        dt1, kv1, thr = time_oracle(wl, k_h, v_h, S, wl.B, sc_h)
        reps = int(min(max(1, np.ceil(10.0 / max(dt1, 1e-3))), max(1, 30.0 // max(dt1, 1e-3))))
        dt, kvb = 0.0, 0
        for _ in range(reps):
            d_, k_, thr = time_oracle(wl, k_h, v_h, S, wl.B, sc_h)
            dt += d_
            kvb += k_
        cpu = {"value": round(kvb / dt / 1e9, 3), "unit": "GB/s", "cores": thr, "kind": "oracle",
               "sample": f"{reps} pass(es) over all {wl.B} sequences, every head, split_kv={S}; {dt:.1f} s fp64",
               "seconds": round(dt, 3)}

    clocks = clk.summary() if not args.no_clocks else None
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": data_text(wl),
        "config": {"workload": args.workload, "B": wl.B, "Sq": wl.Sq, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
                   "page_size": wl.page_size, "num_pages": wl.num_pages, "seq_len": int(wl.seq_lens.max()),
                   "kv_dtype": wl.kv_dtype or wl.dtype, "split_kv": S, "variant": args.variant,
                   "l2": l2_text(wl),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "pct_of_peak": round(100.0 * value / ws / peak, 2),
        "bytes_per_step": ab,
        "roofline": roofline,
        "tflops": round(causal_flops(wl) * ws / (ms_step * 1e-3) / 1e12, 2),
        "kernel_tflops": round(causal_flops(wl) / (fwd_ms * 1e-3) / 1e12, 2),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * (2 if S > 1 else 1),
        "timing": {"protocol": f"{max(args.warmup, 3)} warm-up steps, then the {K} timed steps in "
                               f"{len(batch_sizes(K))} batches of {batch_sizes(K)} steps, CUDA events per batch; "
                               "ms_per_step = median over batches (rocm-libraries PR #14349, Performance)"},
        "clocks": clocks,
    }
    if hot:
        line["hot"] = hot
    if extras:
        line.update(extras)
        line["extras_note"] = ("over2gib, over2gib_same_shape and prefill: further workloads timed in the same run "
                               "with the same protocol; value, roofline and gpu_launches cover the headline "
                               "workload only")
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- variable-length batch
def varlen_bytes(wl) -> dict:
    """Bytes a mixed step must move at least: every valid K and V token once per kv head, q, out,
    page ids, q_start."""
    L = wl.seq_lens.astype(np.int64)
    kv = int(L.sum()) * wl.Hkv * wl.D * wl.esize * 2
    q = wl.Sq * wl.Hq * wl.D * wl.esize
    ids = int(wl.nblk().sum()) * 4 + (2 * wl.B + 1) * 4
    return {"kv": kv, "q": q, "out": q, "ids": ids, "total": kv + 2 * q + ids}


def varlen_flops(wl) -> float:
    """Useful flops: 4 D per (query row, valid key) pair, causal reach with each sequence's offset."""
    pairs = 0
    for b in range(wl.B):
        n = int(wl.q_start[b + 1] - wl.q_start[b])
        L = int(wl.seq_lens[b])
        qoff = (L - n) if wl.q_offset is None else int(wl.q_offset[b])
        reach = np.clip(qoff + np.arange(n) + 1, 0, L) if wl.causal else np.full(n, L)
        pairs += int(reach.sum())
    return 4.0 * wl.D * pairs * wl.Hq


def run_varlen(args, ws, rank, local):
    """The mixed decode + prefill batch through paged_attn_fwd_varlen_overlap: the host-side hint
    (the batch's work split, from its host arrays as a serving scheduler holds them) lets the tcgen05
    kernel (prefill chunks) and the one-grid kernel (decode sequences) run side by side.  For
    context the plain call (the two kernels one after the other) and the same batch as two uniform
    launches are timed too."""
    import torch
    import paged_kv_cache_201_gb300 as pa
    from paged_kv_cache_201_gb300 import workloads as W
    import oracle

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load_library()
    wl = build_workload(args.workload)
    S = args.split_kv or 1
    q = W.host_to_torch(wl.q, wl.dtype).to(dev)
    k, v = W.fill_device_cache(wl, dev)
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    qs = torch.from_numpy(wl.q_start).to(dev)
    qo = torch.from_numpy(wl.q_offset).to(dev)
    T, Hq, D = wl.Sq, wl.Hq, wl.D
    out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    po = torch.empty((S, T, Hq, D), dtype=torch.float32, device=dev) if S > 1 else None
    pl = torch.empty((S, T, Hq), dtype=torch.float32, device=dev) if S > 1 else None
    stream = torch.cuda.current_stream(dev)

    def make_hint():
        return pa.paged_attn_varlen_hint(wl.q_start, wl.seq_lens, wl.q_offset, wl.causal, Hq, wl.Hkv, D,
                                         pa.PA_BF16 if wl.dtype == "bf16" else pa.PA_F16)

    hint = None if args.no_overlap else make_hint()

    def step(h=hint):
        if S == 1:
            pa.paged_attn_fwd_varlen(q, k, v, bt, sl, qs, wl.causal, qo, 1, wl.scale, out, lse, stream, hint=h)
        else:
            pa.paged_attn_fwd_varlen(q, k, v, bt, sl, qs, wl.causal, qo, S, wl.scale, po, pl, stream, hint=h)
            pa.paged_attn_combine(po, pl, out, lse, stream)

    def timed(fn, K):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        return timed_batches([fn], K, stream)[0]

    K = args.steps
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        ms_local = timed(step, K)
    ms_step = max_over_ranks(ms_local, ws, dev)
    flags = pa.paged_attn_last_error_word()
    if flags:
        raise RuntimeError(f"device error word {flags:#x} during the bench")

    # the same batch as two uniform launches: decode sequences (one token) and prefill chunks
    pre = np.nonzero(np.diff(wl.q_start) > 1)[0]
    dec = np.nonzero(np.diff(wl.q_start) == 1)[0]
    assert len(pre) + len(dec) == wl.B and (len(pre) == 0 or pre.max() < dec.min())
    n_pre = len(pre)
    sq_pre = int(wl.q_start[1] - wl.q_start[0]) if n_pre else 0
    assert all(int(wl.q_start[b + 1] - wl.q_start[b]) == sq_pre for b in pre)
    t_pre = n_pre * sq_pre
    q_pre = q[:t_pre].view(n_pre, sq_pre, Hq, D)
    q_dec = q[t_pre:].view(len(dec), 1, Hq, D)
    o_pre = out[:t_pre].view(n_pre, sq_pre, Hq, D)
    o_dec = out[t_pre:].view(len(dec), 1, Hq, D)
    l_pre = lse[:t_pre].view(n_pre, sq_pre, Hq)
    l_dec = lse[t_pre:].view(len(dec), 1, Hq)

    def two_launch():
        pa.paged_attn_fwd(q_pre, k, v, bt[:n_pre], sl[:n_pre], wl.causal, qo[:n_pre], 1, wl.scale, o_pre, l_pre, stream)
        pa.paged_attn_fwd(q_dec, k, v, bt[n_pre:], sl[n_pre:], wl.causal, qo[n_pre:], 1, wl.scale, o_dec, l_dec, stream)

    ms_two = timed(two_launch, max(10, K // 4)) if S == 1 else None
    ms_plain = timed(lambda: step(None), max(10, K // 4)) if hint is not None else None

    ab = varlen_bytes(wl)
    fl = varlen_flops(wl)
    peaks = measured_peaks()
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    achieved = ab["total"] / (ms_local * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "paged_attn_mma_varlen_kernel", "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "kernel_ms": round(ms_local, 5), **traffic_fields("paged_attn_mma_varlen_kernel", args.workload, S),
                "tensor_side": {"achieved_tflops": round(fl / (ms_local * 1e-3) / 1e12, 1)}}

    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (q, bt, sl, qs, qo)]
        po_e = torch.empty_like(po) if S > 1 else None
        pl_e = torch.empty_like(pl) if S > 1 else None

        def call(ins, outs, st):
            qd, btd, sld, qsd, qod = ins
            od, ld = outs
            h = None if args.no_overlap else make_hint()  # the hint from this step's host arrays
            if S == 1:
                pa.paged_attn_fwd_varlen(qd, k, v, btd, sld, qsd, wl.causal, qod, 1, wl.scale, od, ld, st, hint=h)
            else:
                pa.paged_attn_fwd_varlen(qd, k, v, btd, sld, qsd, wl.causal, qod, S, wl.scale, po_e, pl_e, st, hint=h)
                pa.paged_attn_combine(po_e, pl_e, od, ld, st)

        pipe = PipelinedE2E(host_in, lambda j: [torch.empty_like(t, device=dev) for t in host_in],
                            lambda j: [torch.empty_like(out), torch.empty_like(lse)],
                            lambda j: [torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                                       torch.empty(lse.shape, dtype=lse.dtype).pin_memory()], call, stream)
        for _ in range(3):
            pipe.step()
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ev_ms, e2e_wall_ms = e2e_pipelined_batches(pipe, max(10, K // 4))
        e2e_ms = max_over_ranks(e2e_wall_ms, ws, dev)
        e2e_ev_ms = max_over_ranks(e2e_ev_ms, ws, dev)
        hb, db = pipe.bytes()
        e2e = {"value": round(job_throughput(ab["total"], ws, e2e_ms), 1), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db,
               "timing": E2E_TIMING, "pipelining": E2E_PIPELINING,
               "event_value": round(job_throughput(ab["total"], ws, e2e_ev_ms), 1),
               "event_ms_per_step": round(e2e_ev_ms, 4),
               "api": ("paged_attn_fwd_varlen" if args.no_overlap else
                       "paged_attn_varlen_hint + paged_attn_fwd_varlen_overlap") +
                      " (host q / block table / seq_lens / q_start / q_offset in, host out / lse back)"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # the oracle on the decode sequences (each a batch of one), repeated to >= 10 s (cap 30 s)
        k_h, v_h = host_pools(wl, k, v)
        dims = oracle.make_dims(B=len(dec), Sq=1, Hq=Hq, Hkv=wl.Hkv, D=D, page_size=wl.page_size,
                                bt_stride=wl.W, dtype=wl.dtype, num_pages=wl.num_pages)
        qd = wl.q[t_pre:].reshape(len(dec), 1, Hq, D)

        def one_pass():
            t0 = time.perf_counter()
            oracle.rows(q=qd, k_cache=k_h, v_cache=v_h, block_table=wl.block_table[n_pre:],
                        seq_lens=wl.seq_lens[n_pre:], q_offset=wl.q_offset[n_pre:], causal=wl.causal, dims=dims,
                        scale=wl.scale, split_kv=1, want_split=False)
            return time.perf_counter() - t0

        dt1 = one_pass()
        reps = int(min(max(1, np.ceil(10.0 / max(dt1, 1e-3))), max(1, 30.0 // max(dt1, 1e-3))))
        dt = sum(one_pass() for _ in range(reps))
        kvb = reps * int(wl.seq_lens[n_pre:].astype(np.int64).sum()) * wl.Hkv * D * wl.esize * 2
        cpu = {"value": round(kvb / dt / 1e9, 3), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{reps} pass(es) over the {len(dec)} decode sequences of the batch, every head; "
                         f"{dt:.1f} s fp64", "seconds": round(dt, 3)}

    line = {
        "metric": METRIC,
        "value": round(job_throughput(ab["total"], ws, ms_step), 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": data_text(wl),
        "config": {"workload": args.workload, "B": wl.B, "prefill_sequences": n_pre, "prefill_tokens": sq_pre,
                   "decode_sequences": len(dec), "total_query_tokens": T, "Hq": Hq, "Hkv": wl.Hkv, "D": D,
                   "page_size": wl.page_size, "num_pages": wl.num_pages, "split_kv": S, "l2": l2_text(wl),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "bytes_per_step": ab,
        "flops_per_step": fl,
        "roofline": roofline,
        "api": "paged_attn_fwd_varlen" if hint is None else "paged_attn_fwd_varlen_overlap",
        "overlap_sms": None if hint is None else pa.paged_attn_varlen_overlap_share(
            hint, torch.cuda.get_device_properties(dev).multi_processor_count, Hq, wl.Hkv, D,
            pa.PA_BF16 if wl.dtype == "bf16" else pa.PA_F16),
        "plain_call": None if ms_plain is None else {
            "ms_per_step": round(ms_plain, 5),
            "how": "paged_attn_fwd_varlen: the same call with its two kernels one after the other on one stream"},
        "two_launch": None if ms_two is None else {
            "ms_per_step": round(ms_two, 5),
            "how": "the same batch as paged_attn_fwd on the prefill chunks (tcgen05 kernel) then on the "
                   "decode sequences (decode kernel), same stream"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * (2 + (1 if S > 1 else 0)),  # tcgen05 + one-grid kernel (+ the combine)
        "clocks": clk.summary() if not args.no_clocks else None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- reference arm (the oracle)
def run_reference(args, ws, rank, local):
    if rank != 0:
        return
    import torch
    from paged_kv_cache_201_gb300 import workloads as W
    import oracle

    wl = build_workload(args.workload, args.batch)
    S = args.split_kv or wl.split_kv[0]
    sc_h = (wl.k_scale, wl.v_scale) if wl.kv_dtype is not None else None
    if wl.k_cache is not None:
        k_h, v_h = wl.k_cache, wl.v_cache
    else:
        dev = torch.device("cuda", local) if torch.cuda.is_available() else None
        if dev is None:
            print(json.dumps({"impl": "reference", "unavailable": "the 2-GiB pools are drawn on a CUDA device"}))
            return
        if wl.kv_dtype is not None:
            k, v, ks, vs = W.fill_device_cache_q8(wl, dev)
            sc_h = (ks.cpu().numpy(), vs.cpu().numpy())
            del ks, vs
        else:
            k, v = W.fill_device_cache(wl, dev)
        k_h, v_h = host_pools(wl, k, v)
        del k, v
    if wl.q_start is not None:
        # a variable-length batch: sample its first 4 one-token (decode) sequences, each a batch of one
        dec = np.nonzero(np.diff(wl.q_start) == 1)[0][:4]
        t0s = wl.q_start[dec]
        wl = W.Workload(**{**wl.__dict__, "B": len(dec), "Sq": 1, "q": wl.q[t0s].reshape(len(dec), 1, wl.Hq, wl.D),
                           "seq_lens": wl.seq_lens[dec], "block_table": wl.block_table[dec],
                           "q_offset": wl.q_offset[dec], "q_start": None})
    n_seq = min(wl.B, 4)
    time_oracle(wl, k_h, v_h, S, 1, sc_h)  # warm-up: page in the pools and the library
    times, kv = [], 0
    for _ in range(min(args.steps, 20)):
        dt, kv, thr = time_oracle(wl, k_h, v_h, S, n_seq, sc_h)
        times.append(dt)
    ms = float(np.mean(times)) * 1e3
    value = kv / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": len(times),
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": data_text(wl),
        "config": {"workload": args.workload, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
                   "page_size": wl.page_size, "split_kv": S, "sample_sequences": n_seq},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"first {n_seq} of {wl.B} sequences per step, every head"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, ws, rank, local)
    elif args.workload == "mixed_decode_prefill":
        run_varlen(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
