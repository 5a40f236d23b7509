#!/usr/bin/env python
"""Benchmark: sparse paged decode attention on the Qwen3-8B-shaped workload.

One step is one pass of the hot path over one batch (B = 64 sequences, 32 query
/ 8 KV heads, head dim 128, contexts 8K..16K, page size 16, budget 64 pages),
timed as one sparse_decode_step call (the three kernels chained row by row):

  f1-a4  the step's new token appended to each sequence's cache with the
      summary of its page rebuilt (f1, by the scoring pass itself; the a1
      summaries of the rest of the cache are resident), upper-bound scores of
      every page and the top-k budget,
  a5-a6  sparse attention over the selected pages (split-K where rows are few,
      fused merge),
  a7  dense_verify_attn of k+1 = 7 drafted positions over the full cache.

The headline metric is sparse decode-attention tokens/s (B tokens per pass of
f1 and a2-a6); `roofline` is that whole step against the measured HBM copy peak,
over the bytes the method must move (selected K/V tokens, every page summary,
q / o / lse, and the append).  a7 is timed in the same steps (`dense_verify`).
Each kernel is timed with CUDA events on the launching stream; L2 is evicted
between timed passes (a 512 MiB read, outside the events; a write flush would
leave ~L2-size of dirty lines to be written back during the next timed kernel).
The KV cache and the page summaries are resident in HBM (they are the cache);
e2e adds, per step, the host->device copy of the step's inputs (q, the new
token's K / V, seq_lens, page_table), staged in one pinned buffer, and the copy
of o and lse back, one copy each way.

`configs` measures every workload shape of the sweep the same way (tiny, the
Qwen3-1.7B shape with planted retrieval tokens, the Qwen3-8B shape, the
page-size sweep at 16 / 32 / 64, the long-tail batch with split-K), the dense
T = 1 decode beside the tiny and long-tail ones, the retrieval recall of the
selection where tokens are planted, a parity check of sampled sequences against
the fp64 oracle and the oracle's own time on those sequences.

--impl reference times the fp64 CPU oracle (there is no other reference
implementation of this path) on the same workload and metric.
--gpus N without a launcher re-runs this script under torch.distributed.run with
N processes (independent replicas, one per GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_decode_pages_gb300 import workloads as wl  # noqa: E402

METRIC = "sparse decode-attn tokens/s and HBM GB/s (% of roofline), Qwen3-8B shape"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 512 << 20  # read between timed passes: evicts L2 (129 MB) and leaves it clean
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "sparse_attention_decode_pages_gb300", "csrc")
# sources of the kernels whose DRAM traffic profiles/traffic.json records
ATTN_SOURCES = ["common.cuh", "kernels.h", "attn.cuh", "attn_sparse.cu"]
STEP_SOURCES = ["common.cuh", "kernels.h", "attn.cuh", "attn_sparse.cu", "score_select.cu", "spd_api.cu"]
# the workloads of the sweep: (name, page size, dense T = 1 decode beside the sparse step)
CONFIGS = [("tiny", None, True), ("q17b", None, False), ("q8b", None, False), ("sweep", 16, False),
           ("sweep", 32, False), ("sweep", 64, False), ("longtail", None, True)]


def source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(key, files):
    """DRAM bytes per launch recorded by an ncu capture, if the sources are unchanged since."""
    try:
        with open(TRAFFIC_FILE) as fh:
            ent = json.load(fh).get(key)
        if ent and ent.get("source_hash") == source_hash(files):
            return ent["bytes_per_launch"]
    except Exception:
        pass
    return None


def staged(torch, dev, tensors):
    """One device buffer holding the given tensors back to back (each at a 256-byte
    aligned offset), and views of it with their shapes, dtypes and values: a step's
    inputs (or outputs) then move between host and device in one copy."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, off in zip(tensors, offs):
        v = buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank of a multi-GPU run is an independent replica with its own seeded batch."""
    return base_seed + 100 * rank


def max_over_ranks(values, world: int, device):
    """The per-rank timings reduced to their maximum over ranks (the slowest replica
    sets the job's time); a no-op on one rank."""
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tokens_per_s(world: int, batch: int, ms: float) -> float:
    """Whole-job throughput: every replica processes its own batch in `ms`."""
    return world * batch / (ms * 1e-3)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(w, chosen):
    """Bytes the method must move per pass: the valid tokens of the selected pages
    (K and V), every page summary, q / o / lse, and the append (the new token's K
    and V read and written, the older tokens of its page read, its summary written)."""
    ps, D, H_kv = w.page_size, w.D, w.H_kv
    kv = summ = refresh = 0
    for b in range(w.B):
        L = int(w.seq_lens[b])
        summ += w.pages(b) * H_kv * 4 * D
        for h in range(H_kv):
            kv += sum(min(ps, L - p * ps) for p in chosen[b][h]) * 4 * D
        old = (L - 1) - ((L - 1) // ps) * ps
        refresh += H_kv * (2 * D * 2 + old * D * 2 + 4 * D) + H_kv * 2 * D * 2
    qo = w.B * w.H_q * D * 2 * 2 + w.B * w.H_q * 4
    return dict(selected_kv=kv, summaries=summ, q_o_lse=qo, append=refresh,
                attn=kv + qo, score=summ + w.B * w.H_q * D * 2, step=kv + summ + qo + refresh)


def verify_bytes(w, T):
    return sum(int(w.seq_lens[b]) * w.H_kv * 4 * w.D for b in range(w.B)) + w.B * T * w.H_q * w.D * 4


def retrieval_recall(w, sel, nsel):
    """Fraction of the planted retrieval tokens whose page the selection of their
    (sequence, KV head) keeps (every KV head gets the aligned key), or None."""
    hit = tot = 0
    for b in range(w.B):
        for pos in w.planted[b]:
            p = pos // w.page_size
            for h in range(w.H_kv):
                tot += 1
                hit += int(p in set(sel[b, h, : nsel[b, h]].tolist()))
    return None if tot == 0 else hit / tot


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if ts < t0 - 0.06 or ts > t1 + 0.1:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _timed(torch, stream, flush, fn, reps, warmup):
    """Median device time (ms) of fn() between events on the stream, L2 evicted before each."""
    for _ in range(warmup):
        fn()
    out = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        out.append(a.elapsed_time(b))
    return float(np.median(out))


class Case:
    """One workload on the device: its cache, summaries, the step's new token (the K / V
    already at position len - 1, so every pass rewrites the same values and the cache
    stays the same workload), outputs and workspaces."""

    def __init__(self, spd, torch, dev, w):
        self.spd, self.torch, self.dev, self.w = spd, torch, dev, w
        d = self.d = wl.to_device(w, dev)
        self.dims = spd.dims_of(w.B, w.H_q, w.H_kv, w.D, w.page_size, w.max_pages_per_seq, w.num_phys_pages)
        self.summ = torch.empty((w.B, w.H_kv, w.max_pages_per_seq, 2, w.D), dtype=torch.bfloat16, device=dev)
        spd.pages_summarize(self.dims, d["K"], d["page_table"], d["seq_lens"], self.summ)  # prefill
        lens = w.seq_lens.astype(np.int64)
        ph = torch.from_numpy(w.page_table[np.arange(w.B), (lens - 1) // w.page_size].astype(np.int64)).to(dev)
        slot = torch.from_numpy((lens - 1) % w.page_size).to(dev)
        self.k_new = d["K"][ph, :, slot].unsqueeze(1).contiguous()  # [B][1][H_kv][D]
        self.v_new = d["V"][ph, :, slot].unsqueeze(1).contiguous()
        self.sel = torch.empty((w.B, w.H_kv, w.k_max), dtype=torch.int32, device=dev)
        self.nsel = torch.empty((w.B, w.H_kv), dtype=torch.int32, device=dev)
        self.o = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.H_q), dtype=torch.float32, device=dev)
        self.policy = spd.policy_of(w.policy)
        self.ws_step = spd.workspace(spd.spd_sparse_decode_step_workspace_size(self.dims, w.k_max), dev)

    def step(self):
        """One sparse decode step in one call: append, score + select, attention."""
        d = self.d
        self.spd.sparse_decode_step(self.dims, d["K"], d["V"], d["page_table"], d["seq_lens"], self.k_new,
                                    self.v_new, d["q"], self.summ, self.policy, self.sel, self.nsel,
                                    self.w.k_max, self.o, self.ws_step, lse=self.lse)

    def chosen(self):
        n, s = self.nsel.cpu().numpy(), self.sel.cpu().numpy()
        return [[s[b, h, : n[b, h]].tolist() for h in range(self.w.H_kv)] for b in range(self.w.B)], s, n


def _sample(w, k=2):
    """Sequences checked against (and timed with) the oracle: the first and the last."""
    return sorted({0, w.B - 1})[:k]


def oracle_sample(w, sel, nsel, o, lse, dense=None):
    """Parity of sampled sequences against the fp64 oracle, and the oracle's time on them.

    Selection: the share of sampled (sequence, KV head) rows whose page set equals the
    oracle's.  Attention: the oracle over the GPU's own selection (so the numbers
    measure the attention arithmetic, not a tie in the selection).  The CPU time is
    scores + selection + sparse attention of the sampled sequences, one thread each,
    summaries precomputed."""
    import oracle
    seqs = _sample(w)
    n = len(seqs)
    summ = oracle.summarize(w, seqs=seqs, threads=n)
    t0 = time.perf_counter()
    sc = oracle.scores(w, summ, seqs=seqs, threads=n)
    sel_r, nsel_r = oracle.select(w, sc, seqs=seqs, threads=n)
    o_r, lse_r = oracle.sparse_attn(w, sel_r, nsel_r, seqs=seqs, threads=n)
    el = time.perf_counter() - t0
    same = sum(int(nsel[b, h] == nsel_r[b, h] and np.array_equal(sel[b, h, : nsel[b, h]], sel_r[b, h, : nsel_r[b, h]]))
               for b in seqs for h in range(w.H_kv))
    o_g, lse_g = oracle.sparse_attn(w, sel, nsel, seqs=seqs, threads=n)
    err = np.abs(o[seqs].astype(np.float64) - o_g[seqs])
    res = {"sequences": seqs, "selection_rows_identical": same / (n * w.H_kv),
           "o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
           "lse_max_abs": float(np.max(np.abs(lse[seqs] - lse_g[seqs]))),
           "cpu_baseline": {"value": n / el, "unit": "tokens/s", "cores": n, "kind": "oracle",
                            "sample": f"scores + selection + sparse attention of sequences {seqs}"}}
    if dense is not None:
        o_d, lse_d = dense
        q1 = np.ascontiguousarray(w.q.reshape(w.B, 1, w.H_q, w.D))
        t0 = time.perf_counter()
        ov_r, lv_r = oracle.verify(w, 1, q=q1, seqs=seqs, threads=n)
        el = time.perf_counter() - t0
        e = np.abs(o_d[seqs].astype(np.float64) - ov_r[seqs, 0])
        res["dense_t1"] = {"o_max_abs": float(e.max()), "o_mean_abs": float(e.mean()),
                           "lse_max_abs": float(np.max(np.abs(lse_d[seqs] - lv_r[seqs, 0]))),
                           "cpu_baseline": {"value": n / el, "unit": "tokens/s", "cores": n, "kind": "oracle",
                                            "sample": f"dense attention of sequences {seqs}"}}
    return res


def measure_config(spd, torch, dev, name, ps, dense, flush, peak, reps, warmup, stream):
    """The sparse step (and the dense T = 1 decode) of one workload of the sweep."""
    w = wl.named(name, ps)
    c = Case(spd, torch, dev, w)
    ms = _timed(torch, stream, flush, c.step, reps, warmup)
    torch.cuda.synchronize()
    if spd.spd_device_status(clear=True):
        raise RuntimeError(f"device status set in the {name} sweep")
    chosen, sel, nsel = c.chosen()
    nb = algorithmic_bytes(w, chosen)
    gbs = nb["step"] / (ms * 1e-3) / 1e9
    res = {"name": name if ps is None else f"{name} ps{ps}",
           "workload": f"B={w.B}, Hq/Hkv={w.H_q}/{w.H_kv}, D={w.D}, ps={w.page_size}, "
                       f"len {int(w.seq_lens.min())}..{int(w.seq_lens.max())}, budget {w.policy.mode}"
                       f" (mean {float(nsel.mean()):.1f} pages), sink {w.policy.sink_pages} + local "
                       f"{w.policy.local_pages}",
           "sparse_step": {"us": ms * 1e3, "tokens_per_s": w.B / (ms * 1e-3), "gb_s": gbs, "frac": gbs / peak,
                           "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS, "bytes": nb["step"],
                           "summary_share": nb["summaries"] / nb["step"]},
           "recall_planted": retrieval_recall(w, sel, nsel)}
    o_h, lse_h = c.o.float().cpu().numpy(), c.lse.cpu().numpy()
    dense_out = None
    if dense:
        ov = torch.empty((w.B, 1, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
        lv = torch.empty((w.B, 1, w.H_q), dtype=torch.float32, device=dev)
        q1 = c.d["q"].view(w.B, 1, w.H_q, w.D)
        wsv = spd.workspace(spd.spd_dense_verify_workspace_size(c.dims, 1, 0), dev)
        msd = _timed(torch, stream, flush, lambda: spd.dense_verify_attn(
            c.dims, 1, q1, c.d["K"], c.d["V"], c.d["page_table"], c.d["seq_lens"], ov, wsv, lse=lv), reps, warmup)
        vb = verify_bytes(w, 1)
        res["dense_t1"] = {"us": msd * 1e3, "tokens_per_s": w.B / (msd * 1e-3), "gb_s": vb / (msd * 1e-3) / 1e9,
                           "frac": vb / (msd * 1e-3) / 1e9 / peak, "bytes": vb}
        dense_out = (ov[:, 0].float().cpu().numpy(), lv[:, 0].cpu().numpy())
    if spd.spd_device_status(clear=True):
        raise RuntimeError(f"device status set in the {name} sweep")
    res["oracle"] = oracle_sample(w, sel, nsel, o_h, lse_h, dense_out)
    del c
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import sparse_attention_decode_pages_gb300 as spd

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    # Each rank is an independent replica with its own seeded batch.
    spec = wl.spec(args.config, args.page_size)
    spec.seed = replica_seed(spec.seed, rank)
    if args.batch:
        spec.B = args.batch
    w = wl.make(spec)
    T = w.T or 7
    if w.q_verify is None:
        rng = np.random.default_rng(spec.seed + 7)
        w.q_verify = wl.f32_to_bf16_bits(rng.standard_normal((w.B, T, w.H_q, w.D)).astype(np.float32))
    c = Case(spd, torch, dev, w)
    d, dims, summ, k_max = c.d, c.dims, c.summ, w.k_max
    # the step's inputs and outputs each in one device buffer (one copy each way in e2e)
    inp_d, (d["q"], d["seq_lens"], d["page_table"], c.k_new, c.v_new) = staged(
        torch, dev, [d["q"], d["seq_lens"], d["page_table"], c.k_new, c.v_new])
    out_d, (c.o, c.lse) = staged(torch, dev, [c.o, c.lse])
    ov = torch.empty((w.B, T, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
    lsev = torch.empty((w.B, T, w.H_q), dtype=torch.float32, device=dev)
    ws_sel = spd.workspace(spd.spd_score_select_workspace_size(dims), dev)
    ws_attn = spd.workspace(spd.spd_sparse_decode_workspace_size(dims, k_max, args.splits), dev)
    ws_ver = spd.workspace(spd.spd_dense_verify_workspace_size(dims, T, args.vsplits), dev)
    flush_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        """Evicts L2 by reading a buffer 4x its size (a write would leave dirty lines
        to be written back during the next timed kernel)."""
        flush_buf.sum()

    stream = torch.cuda.current_stream(dev)

    def sparse_pass(ev=None):
        if ev is None and args.splits == 0:
            c.step()  # the whole step in one call: append, score + select and attention chained
            return
        if ev:
            ev[0].record(stream)
        # f1 + a2-a4: the step's token appended (its page's summary rebuilt) by the
        # scoring pass itself, then the selection
        spd.pages_append_score_select(dims, d["K"], d["V"], d["page_table"], d["seq_lens"], c.k_new, c.v_new,
                                      d["q"], summ, c.policy, c.sel, c.nsel, k_max, ws_sel)
        if ev:
            ev[2].record(stream)
        spd.sparse_decode_attn(dims, d["q"], d["K"], d["V"], d["page_table"], d["seq_lens"], c.sel,
                               c.nsel, k_max, c.o, ws_attn, lse=c.lse, num_splits=args.splits)
        if ev:
            ev[3].record(stream)

    def verify_pass(ev=None):
        if ev:
            ev[0].record(stream)
        spd.dense_verify_attn(dims, T, d["q_verify"], d["K"], d["V"], d["page_table"],
                              d["seq_lens"], ov, ws_ver, lse=lsev, num_splits=args.vsplits)
        if ev:
            ev[1].record(stream)

    for _ in range(args.warmup):
        sparse_pass()
        flush()
        verify_pass()
        flush()
    torch.cuda.synchronize()
    status = spd.spd_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} after warm-up")

    chosen, sel_host, nsel_host = c.chosen()
    o_host, lse_host = c.o.float().cpu().numpy(), c.lse.cpu().numpy()
    nbytes = algorithmic_bytes(w, chosen)
    vbytes = verify_bytes(w, T)

    # Two passes over the same K steps.  Pass A times each step as a whole (events
    # only at its ends, so the step's kernels overlap their launches as they do
    # in use); pass B puts events between the kernels (which serialises them)
    # for the per-kernel breakdown.
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evs = [[torch.cuda.Event(enable_timing=True) if k != 1 else None for k in range(4)] for _ in range(args.steps)]
    vevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush()
        sevs[i][0].record(stream)
        sparse_pass()
        sevs[i][1].record(stream)
        flush()
        verify_pass(vevs[i])
    for i in range(args.steps):
        flush()
        sparse_pass(evs[i])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    status = spd.spd_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} in the timed region")

    t_sel = [e[0].elapsed_time(e[2]) for e in evs]
    t_att = [e[2].elapsed_time(e[3]) for e in evs]
    t_step = [e[0].elapsed_time(e[1]) for e in sevs]
    t_step_serial = [e[0].elapsed_time(e[3]) for e in evs]
    t_ver = [e[0].elapsed_time(e[1]) for e in vevs]
    ms_step = float(np.mean(t_step))
    ms_ver = float(np.mean(t_ver))
    ms_att = float(np.mean(t_att))
    ms_sel = float(np.mean(t_sel))

    # e2e: the same sparse pass through the C ABI with host buffers: the step's inputs
    # (q, seq_lens, page_table, the new token's K / V) staged in one pinned buffer and
    # copied in, o and lse copied out.
    inp_h = inp_d.cpu().pin_memory()
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        inp_d.copy_(inp_h, non_blocking=True)
        sparse_pass()
        out_h.copy_(out_d, non_blocking=True)
        eb.record(stream)
        eb.synchronize()
        if i >= args.warmup:
            e2e_ms.append(ea.elapsed_time(eb))
    h2d = inp_h.numel()  # bytes, with each input padded to 256
    d2h = out_h.numel()

    nxt = None if args.no_next else next_rows(spd, torch, w, d, dims, summ, stream, flush, peak_of=hbm_peak,
                                              reps=max(10, min(args.steps, 50)), warmup=args.warmup)

    # max over ranks
    ms_step, ms_ver, ms_e2e, ms_att, ms_sel = max_over_ranks(
        [ms_step, ms_ver, float(np.mean(e2e_ms)), ms_att, ms_sel], world, dev)

    peak, peak_src = hbm_peak()
    peak_note = (f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, copy peak)" if peak_src == "measured"
                 else "fallback 6.8 TB/s")
    step_gbs = nbytes["step"] / (ms_step * 1e-3) / 1e9
    att_gbs = nbytes["attn"] / (ms_att * 1e-3) / 1e9
    sel_gbs = (nbytes["score"] + nbytes["append"]) / (ms_sel * 1e-3) / 1e9
    ver_gbs = vbytes / (ms_ver * 1e-3) / 1e9

    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = []
        for name, ps, dense in CONFIGS:
            if name == args.config and ps == args.page_size:
                # the headline workload, measured above; its oracle sample here
                configs.append({"name": name, "workload": "the headline workload (config)",
                                "sparse_step": {"us": ms_step * 1e3, "tokens_per_s": w.B / (ms_step * 1e-3),
                                                "gb_s": step_gbs, "frac": step_gbs / peak,
                                                "frac_of_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS,
                                                "bytes": nbytes["step"],
                                                "summary_share": nbytes["summaries"] / nbytes["step"]},
                                "dense_verify_t7": {"us": ms_ver * 1e3, "tokens_per_s": w.B * T / (ms_ver * 1e-3),
                                                    "gb_s": ver_gbs, "frac": ver_gbs / peak},
                                "recall_planted": retrieval_recall(w, sel_host, nsel_host),
                                "oracle": oracle_sample(w, sel_host, nsel_host, o_host, lse_host)})
                continue
            configs.append(measure_config(spd, torch, dev, name, ps, dense, flush, peak, reps=20,
                                          warmup=3, stream=stream))

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, T)
        line = {
            "metric": METRIC,
            "value": job_tokens_per_s(world, w.B, ms_step),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded; shapes of the Qwen3-8B rollout workload)",
            "config": {
                "workload": f"{args.config}: B={w.B}, Hq/Hkv={w.H_q}/{w.H_kv}, D={w.D}, "
                            f"ps={w.page_size}, len {int(w.seq_lens.min())}..{int(w.seq_lens.max())}, "
                            f"budget {w.policy.fixed_pages if w.policy.mode == 'fixed' else w.policy.mode} pages, "
                            f"sink 1 + local {w.policy.local_pages}; verify T={T}",
                "global_batch": world * w.B,
                "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                "l2": "evicted between timed passes by reading a 512 MiB buffer (outside the events)",
                "timing": "value and roofline from whole-step events around sparse_decode_step (its kernels "
                          "chained row by row); the per-kernel breakdown from a second pass of the separate "
                          "calls with events between them",
                "splits": args.splits, "verify_splits": args.vsplits,
            },
            # the gated quantity: score + select + sparse attention + merge (with the step's
            # append), over the bytes the method must move
            "roofline": {"bound": "hbm", "kernel": "sparse_decode_step (append + score + select + sparse "
                                                  "attention + merge, chained)",
                         "achieved": step_gbs, "peak": peak, "unit": "GB/s", "frac": step_gbs / peak,
                         "frac_of_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS,
                         "traffic": recorded_traffic(f"sparse_decode_step/{args.config}", STEP_SOURCES),
                         "algorithmic_bytes": nbytes["step"],
                         "bytes": {k: nbytes[k] for k in ("selected_kv", "summaries", "q_o_lse", "append")},
                         "peak_source": peak_note},
            "kernels": {
                "sparse_attn": {"kernel": "attn_kernel (sparse, fused merge), separate call", "ms": ms_att,
                                "achieved": att_gbs, "frac": att_gbs / peak, "unit": "GB/s",
                                "algorithmic_bytes": nbytes["attn"],
                                "traffic": recorded_traffic(f"sparse_decode_attn/{args.config}", ATTN_SOURCES)},
                "append_score_select": {"kernel": "score_select_kernel + select_kernel, separate call",
                                        "ms": ms_sel, "achieved": sel_gbs, "frac": sel_gbs / peak,
                                        "unit": "GB/s", "algorithmic_bytes": nbytes["score"] + nbytes["append"]},
            },
            "step_ms": {"whole_step": ms_step, "serialised_step": float(np.mean(t_step_serial)),
                        "f1_a2_a4_append_score_select": ms_sel, "a5_a6_sparse_attn": ms_att},
            "dense_verify": {"tokens_per_s": world * w.B * T / (ms_ver * 1e-3), "ms": ms_ver,
                             "achieved_gbs": ver_gbs, "frac": ver_gbs / peak, "bytes": vbytes,
                             "tflops": 4.0 * sum(int(w.seq_lens[b]) for b in range(w.B)) * w.H_q * T * w.D
                             / (ms_ver * 1e-3) / 1e12},
            "e2e": {"value": job_tokens_per_s(world, w.B, ms_e2e), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms": ms_e2e},
            # pass A per step: append + score (1), select (1), sparse attention with its
            # fused merge (1), dense verification (1); pass B: the first three again
            "gpu_launches": args.steps * 7,
            "clocks": clocks,
            "wall_s_timed_region": t1 - t0,
            "cpu_baseline": cpu,
            "configs": configs,
            "next_rows": nxt,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def next_rows(spd, torch, w, d, dims, summ, stream, flush, peak_of, reps, warmup):
    """The rows after the core path, measured on the same workload after its timed region:
    exact speculative sampling (B sequences, k = 6, Qwen3's vocabulary), top-p page
    selection, and the S3R round as CUDA graphs against the same calls made eagerly."""
    import dataclasses
    dev = d["q"].device
    peak, _ = peak_of()
    k = 6
    res = {}
    # f2: speculative sampling
    sp = wl.spec_inputs(B=w.B, k=k)
    P = torch.from_numpy(sp["p"]).to(dev)
    Q = torch.from_numpy(sp["q"]).to(dev)
    Dr = torch.from_numpy(sp["draft"]).to(dev)
    Ua = torch.from_numpy(sp["u_acc"]).to(dev)
    Ur = torch.from_numpy(sp["u_res"]).to(dev)
    na = torch.empty(w.B, dtype=torch.int32, device=dev)
    tk = torch.empty((w.B, k + 1), dtype=torch.int32, device=dev)
    ms = _timed(torch, stream, flush, lambda: spd.spec_accept(P, Q, Dr, Ua, Ur, na, tk), reps, warmup)
    nacc = na.cpu().numpy()
    n = sp["p"].shape[-1]
    rows = sum(2 if a < k else 1 for a in nacc)   # residual rows read p and q; the bonus row q only
    byts = rows * n * 4 + w.B * k * 16
    res["f2_spec_accept"] = {"us": ms * 1e3, "bytes": byts, "achieved_gbs": byts / (ms * 1e-3) / 1e9,
                             "frac": byts / (ms * 1e-3) / 1e9 / peak, "k": k, "n_vocab": n,
                             "mean_accepted": float(nacc.mean())}
    del P, Q
    # f3: top-p selection (scores + select) against the fixed top-k budget
    pol = dataclasses.replace(w.policy, mode="top_p", top_p=0.9, score_scale=1.0 / math.sqrt(w.D))
    k_max = w.max_pages_per_seq
    sel = torch.empty((w.B, w.H_kv, k_max), dtype=torch.int32, device=dev)
    nsel = torch.empty((w.B, w.H_kv), dtype=torch.int32, device=dev)
    ws = spd.workspace(spd.spd_score_select_workspace_size(dims), dev)
    ms = _timed(torch, stream, flush, lambda: spd.pages_score_select(dims, d["q"], summ, d["seq_lens"], pol, sel,
                                                                     nsel, k_max, ws), reps, warmup)
    res["f3_top_p_score_select"] = {"us": ms * 1e3, "top_p": 0.9, "mean_pages": float(nsel.float().mean()),
                                    "max_pages": int(nsel.max())}
    # f4: one S3R round (6 draft steps; verification of 7 positions + sampling) as graphs vs eager
    r = wl.round_inputs(w, k=k, n_vocab=n)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    lens = i32(r["seq_lens"])
    qd, kd, vd = bf(r["q_draft"]), bf(r["k_draft"]), bf(r["v_draft"])
    qv, kv, vv = bf(r["q_verify"]), bf(r["k_verify"]), bf(r["v_verify"])
    smp = dict(p_draft=f32(r["p"]), q_target=f32(r["q"]), draft_tokens=i32(r["draft"]), u_acc=f32(r["u_acc"]),
               u_res=f32(r["u_res"]), n_accepted=torch.zeros(w.B, dtype=torch.int32, device=dev),
               tokens=torch.zeros((w.B, k + 1), dtype=torch.int32, device=dev))
    kx = w.k_max
    sel = torch.empty((w.B, w.H_kv, kx), dtype=torch.int32, device=dev)
    nsel = torch.empty((w.B, w.H_kv), dtype=torch.int32, device=dev)
    od = torch.empty((k, w.B, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
    ov = torch.empty((w.B, k + 1, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
    ws_sel = spd.workspace(spd.spd_score_select_workspace_size(dims), dev)
    ws_sp = spd.workspace(spd.spd_sparse_decode_workspace_size(dims, kx, 0), dev)
    ws_ver = spd.workspace(spd.spd_dense_verify_workspace_size(dims, k + 1, 0), dev)
    K, V, pt = d["K"], d["V"], d["page_table"]

    def eager_draft():
        for s_ in range(k):
            spd.kv_append_refresh(dims, 1, K, V, pt, lens[s_], kd[s_], vd[s_], summ)
            spd.pages_score_select(dims, qd[s_], summ, lens[s_], w.policy, sel, nsel, kx, ws_sel)
            spd.sparse_decode_attn(dims, qd[s_], K, V, pt, lens[s_], sel, nsel, kx, od[s_], ws_sp)

    def eager_verify():
        spd.kv_append_refresh(dims, k + 1, K, V, pt, lens[k], kv, vv, summ)
        spd.dense_verify_attn(dims, k + 1, qv, K, V, pt, lens[k], ov, ws_ver)
        spd.spec_accept(smp["p_draft"], smp["q_target"], smp["draft_tokens"], smp["u_acc"], smp["u_res"],
                        smp["n_accepted"], smp["tokens"])

    rnd = spd.Round(dims, k, K, V, summ, pt, lens, qd, kd, vd, qv, kv, vv, w.policy, kx, sel, nsel, od, ov,
                    ws_sel, ws_sp, ws_ver, sampling=smp)
    e_d = _timed(torch, stream, flush, eager_draft, reps, warmup)
    e_v = _timed(torch, stream, flush, eager_verify, reps, warmup)
    g_d = _timed(torch, stream, flush, lambda: rnd.launch(0, stream), reps, warmup)
    g_v = _timed(torch, stream, flush, lambda: rnd.launch(1, stream), reps, warmup)
    acc = smp["n_accepted"].float().mean().item()
    rnd.close()
    res["f4_s3r_round"] = {"k": k, "draft_graph_ms": g_d, "verify_graph_ms": g_v, "draft_eager_ms": e_d,
                           "verify_eager_ms": e_v, "mean_accepted": acc,
                           "round_tokens_per_s": w.B * (acc + 1) / ((g_d + g_v) * 1e-3),
                           "note": "L2 evicted before each part; the 6 draft steps run back to back inside it"}
    if spd.spd_device_status(clear=True):
        raise RuntimeError("device status set while measuring the next rows")
    return res


def _oracle_sparse_step(w, summ, threads):
    import oracle
    sc = oracle.scores(w, summ, threads=threads)
    sel, nsel = oracle.select(w, sc, threads=threads)
    return oracle.sparse_attn(w, sel, nsel, threads=threads)


def cpu_baseline(w, T, min_seconds=3.0):
    """The fp64 oracle as it stands on the host cores: score + select + sparse attention."""
    import oracle
    threads = os.cpu_count() or 1
    summ = oracle.summarize(w, threads=threads)  # prefill, outside the timing
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_sparse_step(w, summ, threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    t1 = time.perf_counter()
    _oracle_sparse_step(w, summ, 1)  # the same pass on one thread
    el1 = time.perf_counter() - t1
    return {"value": n * w.B / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full passes of scores + selection + sparse attention over the whole "
                      f"batch (B={w.B}); page summaries precomputed once outside the timing",
            "single_thread": {"value": w.B / el1, "unit": "tokens/s", "sample": "one full pass on 1 thread"}}


def run_reference(args):
    """The oracle arm: rank 0 only; every step is one full pass over the batch."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    w = wl.named(args.config, args.page_size)
    threads = os.cpu_count() or 1
    summ = oracle.summarize(w, threads=threads)
    for _ in range(args.warmup):
        _oracle_sparse_step(w, summ, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sparse_step(w, summ, threads)
    el = time.perf_counter() - t0
    value = args.steps * w.B / el
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the Qwen3-8B rollout workload)",
        "config": {"workload": f"{args.config}: B={w.B}, Hq/Hkv={w.H_q}/{w.H_kv}, D={w.D}, "
                               f"ps={w.page_size}", "global_batch": w.B,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} passes of scores + selection + sparse attention "
                                   f"over the whole batch; summaries precomputed"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def replica_launch_cmd(argv, n, port):
    """The command that runs this benchmark as n independent replicas, one process per GPU."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="replicas (one per GPU); without a launcher the "
                                                        "script re-runs itself under torch.distributed.run")
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="q8b", choices=["tiny", "q17b", "q8b", "sweep", "longtail"])
    ap.add_argument("--page-size", type=int, default=None)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--vsplits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the measurements of the rows after the core path")
    ap.add_argument("--no-configs", action="store_true", help="skip the sweep over the other workload shapes")
    ap.add_argument("--batch", type=int, default=0, help="override B (small profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = os.environ.get("WORLD_SIZE")
    if args.gpus > 1 and world is None:
        sys.exit(subprocess.call(replica_launch_cmd(sys.argv[1:], args.gpus, _free_port())))
    if world is not None and int(world) != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; running {world} replicas", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
