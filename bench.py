#!/usr/bin/env python
"""Benchmark of the MLA latent-cache hot path on GB300.

Headline workload (default --workload): sparse prefill over fp8_ds_mla records (T=4096 query
rows, H=16, top-2048 of 65536 records, ~5 % masked), the largest configuration that fits one
GPU.  One step = one mla_sparse_fwd over the whole batch.  The same JSON line carries, under
"per_config", the other workloads of the path, each timed the same way with its own roofline,
end-to-end figure and CPU-oracle baseline:
  decode_bf16_epilogue  mla_q_concat_cache_insert + mla_paged_decode (B=32, q=1, H=16, bf16,
                        seq_lens ~ U[1024, 8192])
  fp8_spec_verify       mla_paged_decode (B=64, q=4 causal, H=16, plain fp8, L ~ U[16k, 128k],
                        split-K + merge)
  ds_mla_h96_decode     mla_paged_decode (B=128, H=96, fp8_ds_mla, L ~ U[8k, 32k])
  sparse_prefill_4M_records  the headline over a 2^22-record pool (2.75 GB, past L2)

Metric: achieved GB/s of algorithmic bytes (entries gathered + query read + output written
(+ lse)), with query-rows/s beside it.  Timing: CUDA events per step after warm-up, L2
flushed (256 MiB write) between steps outside the timed events; max over ranks.  A step's
launches are captured once into a CUDA graph and replayed per timed step (the serving
pattern: no host marshalling between the step's kernels); the attention kernel's own time
(roofline) comes from per-launch events around ordinary calls.  The
headline times exactly --steps steps; each per-config entry times at least --steps steps and
at least --min-ms of GPU time (so that clock samples land under load).
The "e2e" figure goes through the public API with the step's inputs copied from pinned
host memory and its results copied back inside the timed region: the sparse prefill streams
its rows in four chunks (kv_indptr slices) so that copies overlap the kernel; the paged
workloads stage each step's inputs in one pinned buffer and its out + lse in another, and
replay one CUDA graph of the two copies and the calls ("e2e.mode" says which).
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs an independent replica ("replicas only").
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA attention achieved HBM GB/s (% of GB300 peak); query-rows/s at 1 GPU"
WORKLOADS = ("sparse_prefill", "decode_bf16_epilogue", "fp8_spec_verify", "ds_mla_h96_decode")
# the attention kernel each workload times (the profiling hook brackets exactly its launch)
KERNELS = {
    "decode_bf16_epilogue": "mla_paged_tma_kernel<bf16, 16 columns>",
    "sparse_prefill": "mla_ds_kernel<sparse> (gather warps)",
    "fp8_spec_verify": "mla_paged_tma_kernel<fp8, 64 columns>",
    "ds_mla_h96_decode": "mla_ds_kernel<paged>",
}
PAST_L2_RECORDS = 1 << 22


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s (measured burst figure when present)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops"
    except Exception:
        return 1900.0, "fallback"


# ------------------------------------------------------------------------------------ workloads

class Work:
    """Host inputs of one workload plus its byte / row accounting."""

    def __init__(self, name: str, batch: int = 0, records: int = 0):
        from mla_latent_cache_attention_gb300 import synth
        self.name = name
        self.synth = synth
        # batch > 0 keeps the workload's geometry with fewer requests (profiling captures that
        # must stay small); bench lines use the full workload
        kw = dict(B=batch) if batch > 0 else {}
        if name == "decode_bf16_epilogue":
            self.case, self.epi = synth.config1(**kw)
            self.kind = "paged"
        elif name == "sparse_prefill":
            # records > 0: a record pool of that size (2^22 records, 2.75 GB, is past L2, so the
            # gathered records come from DRAM instead of L2)
            kw2 = dict(T=batch) if batch > 0 else {}
            if records > 0:
                kw2["N"] = records
            self.case = synth.config2(**kw2)
            self.kind = "sparse"
        elif name == "fp8_spec_verify":
            self.case = synth.config3(**kw)
            self.kind = "paged"
        elif name == "ds_mla_h96_decode":
            self.case = synth.config4(**kw)
            self.kind = "paged"
        else:
            raise SystemExit(f"unknown workload {name}")
        c = self.case
        if self.kind == "sparse":
            self.attn_bytes = synth.algorithmic_bytes_sparse(c)
            self.rows = c.q.shape[0]
            self.heads = c.q.shape[1]
            self.cfg = dict(workload=name, T=int(c.q.shape[0]), H=int(c.q.shape[1]), records=int(c.records.shape[0]),
                            indices_per_row=2048, masked_frac=0.05, cache="fp8_ds_mla", return_lse=True)
            self.dtype = "fp8_ds_mla: e4m3 codes (kind::f8f6f4) + bf16 rope (kind::f16), fp32 accumulate"
        else:
            self.attn_bytes = synth.algorithmic_bytes_paged(c)
            self.rows = c.seq_lens.size * c.q_len
            self.heads = c.H
            fmtname = {0: "bf16", 1: "fp8", 2: "fp8_ds_mla"}[c.fmt]
            self.cfg = dict(workload=name, B=int(c.seq_lens.size), q_len=c.q_len, H=c.H, cache=fmtname,
                            block_size=int(c.cache.shape[1]), seq_len_lo=int(c.meta["L_lo"]),
                            seq_len_hi=int(c.meta["L_hi"]), max_context=c.max_context, return_lse=c.return_lse)
            self.dtype = {0: "bf16 (kind::f16 MMA, fp32 accumulate)",
                          1: "fp8 e4m3 operands (kind::f8f6f4 MMA, fp32 accumulate)",
                          2: "fp8_ds_mla: e4m3 codes (kind::f8f6f4) + bf16 rope (kind::f16), fp32 accumulate"}[c.fmt]
        # the dense contraction per (query row, head, visible key): 2 * 576 (QK) + 2 * 512 (PV)
        if self.kind == "sparse":
            visible = int(np.count_nonzero((c.indices >= 0) & (c.indices < c.records.shape[0])))
        else:
            L = c.seq_lens.astype(np.int64)
            visible = int(sum(np.clip(L - c.q_len + i + 1, 0, None).sum() for i in range(c.q_len)))
        self.flops = visible * self.heads * (2 * 576 + 2 * 512)
        self.epi_bytes = 0
        if name == "decode_bf16_epilogue":
            B, H = self.epi.ql_nope.shape[:2]
            # epilogue: ql_nope + q_pe + kv_c + k_pe read, cos/sin rows, mqa_q and the entries written
            self.epi_bytes = 2 * (B * H * 576 + B * 576) + B * 64 * 4 + 2 * B * H * 576 + B * 1152
        self.step_bytes = self.attn_bytes + self.epi_bytes


# ------------------------------------------------------------------------------------ GPU arm

def to_dev(a, torch, dev, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(dev)


class GpuRunner:
    def __init__(self, w: Work, dev):
        import torch
        import mla_latent_cache_attention_gb300 as m
        self.torch, self.m, self.w, self.dev = torch, m, w, dev
        c = w.case
        if w.kind == "sparse":
            self.q = to_dev(c.q.view(np.int16), torch, dev).view(torch.bfloat16)
            self.rec = to_dev(c.records, torch, dev)
            self.indptr = to_dev(c.indptr, torch, dev)
            self.indices = to_dev(c.indices, torch, dev)
            self.out = torch.empty((self.q.shape[0], self.q.shape[1], 512), dtype=torch.bfloat16, device=dev)
            self.launches_per_step = 1
        else:
            self.cache = to_dev(c.cache, torch, dev)
            self.bt = to_dev(c.block_table, torch, dev)
            self.sl = to_dev(c.seq_lens, torch, dev)
            if c.fmt == 1:
                self.q = to_dev(c.q, torch, dev)
            else:
                self.q = to_dev(c.q.view(np.int16), torch, dev).view(torch.bfloat16).reshape(c.q.shape[0], c.H, 576)
            self.out = torch.empty((self.q.shape[0], c.H, 512), dtype=torch.bfloat16, device=dev)
            need = m.paged_decode_workspace_size(c.seq_lens.size, c.q_len, c.H, c.max_context)
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            # the attention kernel, and with split-K the scheduler reset and the merge
            self.launches_per_step = 1 + (2 if need > 0 else 0)
            if w.name == "decode_bf16_epilogue":
                e = w.epi
                b16 = lambda a: to_dev(a.view(np.int16), torch, dev).view(torch.bfloat16)
                self.ql, self.qp, self.kvc, self.kpe = b16(e.ql_nope), b16(e.q_pe), b16(e.kv_c), b16(e.k_pe)
                self.slots = to_dev(e.slot_mapping, torch, dev)
                self.pos = to_dev(e.positions, torch, dev)
                self.cs = to_dev(e.cos_sin, torch, dev)
                self.launches_per_step += 1
        self.lse = torch.empty((self.q.shape[0], self.q.shape[1]), dtype=torch.float32, device=dev)

    def step(self):
        m, w, c = self.m, self.w, self.w.case
        if w.kind == "sparse":
            m.sparse_fwd(self.q, self.rec, self.indptr, self.indices, c.softmax_scale, has_invalid=True,
                         out=self.out, return_lse=True, lse=self.lse)
            return
        q = self.q
        if w.name == "decode_bf16_epilogue":
            q = m.q_concat_cache_insert(self.ql, self.qp, self.kvc, self.kpe, self.cache, self.slots,
                                        fmt=c.fmt, positions=self.pos, cos_sin_cache=self.cs, mqa_q=self.q)
        m.paged_decode(q, self.cache, self.bt, self.sl, fmt=c.fmt, q_len=c.q_len, max_context=c.max_context,
                       softmax_scale=c.softmax_scale, q_scale=c.q_scale, k_scale=c.k_scale, out=self.out,
                       return_lse=c.return_lse, workspace=self.ws, lse=self.lse if c.return_lse else None)

    # ---- end-to-end: the per-step inputs come from pinned host memory, the result goes back
    def e2e_setup(self):
        torch, w, c = self.torch, self.w, self.w.case
        pin = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).view(dt) if dt is not None else
                                  torch.from_numpy(np.ascontiguousarray(a))).pin_memory()
        self.copy_s, self.d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        self.comp2_s = torch.cuda.Stream()
        self.e2e_graph = None
        if w.kind == "sparse":
            # the rows stream in chunks: the copies of chunk i + 1 and the results of chunk
            # i - 1 move while chunk i computes (a kv_indptr slice addresses the same kv_indices)
            self.h_in = [(pin(c.q.view(np.int16), torch.bfloat16), self.q), (pin(c.indptr), self.indptr),
                         (pin(c.indices), self.indices)]
            self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
            self.h_lse = torch.empty(self.lse.shape, dtype=self.lse.dtype).pin_memory()
            self.h2d = sum(h.numel() * h.element_size() for h, _ in self.h_in)
            self.d2h = self.h_out.numel() * 2 + self.h_lse.numel() * 4
            self.e2e_mode = f"{self.E2E_CHUNKS} row chunks pipelined over copy / two compute / copy-back streams"
            self.h_ptr = c.indptr.astype(np.int64)
            T = c.q.shape[0]
            # short first and last chunks: the copy-in before the first kernel and the copy-back
            # after the last one are what stays exposed
            cum = np.concatenate([[0], np.cumsum(self.E2E_SPLIT)])
            self.bounds = [int(T * x // cum[-1]) for x in cum]
            return
        # a decode step's inputs (and its out + lse) live in one device buffer each, as a serving
        # loop would stage them: one host -> device and one device -> host copy per step, inside
        # one CUDA graph with the API calls
        names = ["q", "bt", "sl"]
        if w.name == "decode_bf16_epilogue":
            names = ["ql", "qp", "kvc", "kpe", "slots", "pos", "bt", "sl"]
        self.ret_lse = bool(c.return_lse)
        self.h_in_pack, self.d_in_pack = self._pack([(n, getattr(self, n)) for n in names])
        outs = [("out", self.out)] + ([("lse", self.lse)] if self.ret_lse else [])
        self.h_out_pack, self.d_out_pack = self._pack(outs)
        self.h2d = self.h_in_pack.numel()
        self.d2h = self.h_out_pack.numel()
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                self.e2e_direct()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.e2e_direct()
            torch.cuda.synchronize()
            self.e2e_graph = g
            self.e2e_mode = "CUDA graph: one packed input copy, the API calls, one packed result copy"
        except Exception:
            torch.cuda.synchronize()
            self.e2e_mode = "direct API calls, packed copies"

    def _pack(self, named):
        """Rebind each named device tensor to a view of one new device buffer (256-byte aligned
        pieces, same contents) and return (pinned host buffer of the same layout and contents,
        device buffer)."""
        torch = self.torch
        offs, off = [], 0
        for _, t in named:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        dbuf = torch.empty(off, dtype=torch.uint8, device=self.dev)
        hbuf = torch.zeros(off, dtype=torch.uint8).pin_memory()
        for (n, t), o in zip(named, offs):
            nb = t.numel() * t.element_size()
            view = dbuf[o:o + nb].view(t.dtype).view(t.shape)
            view.copy_(t)
            hbuf[o:o + nb].copy_(t.contiguous().view(torch.uint8).reshape(-1).cpu())
            setattr(self, n, view)
        return hbuf, dbuf

    # row chunks in the proportions 1:2:2:2:2:1 over two compute streams; measured e2e (1.78 ms
    # kernel): 1:3:3:1 2758 GB/s, 1:2:2:2:1 2839, 1:2:2:2:2:1 2848, 1:3:3:3:1 2793, 8 equal 2818
    # (one compute stream: 1:3:3:1 2622; with the 2.0 ms kernel equal quarters 2323, 1:3:3:1 2433)
    E2E_SPLIT = (1, 2, 2, 2, 2, 1)
    E2E_CHUNKS = len(E2E_SPLIT)

    def e2e_direct(self):
        self.d_in_pack.copy_(self.h_in_pack, non_blocking=True)
        self.step()
        self.h_out_pack.copy_(self.d_out_pack, non_blocking=True)

    def e2e_step(self):
        torch, m, c = self.torch, self.m, self.w.case
        if self.e2e_graph is not None:
            self.e2e_graph.replay()
            return
        if self.w.kind != "sparse":
            self.e2e_direct()
            return
        cur = torch.cuda.current_stream()
        (hq, _), (hptr, _), (hidx, _) = self.h_in
        self.copy_s.wait_stream(cur)
        self.d2h_s.wait_stream(cur)
        self.comp2_s.wait_stream(cur)
        with torch.cuda.stream(self.copy_s):
            self.indptr.copy_(hptr, non_blocking=True)
        # chunks alternate between two compute streams: the next chunk's CTAs take the SMs that
        # the previous chunk's last rows leave idle
        comp = (cur, self.comp2_s)
        for i in range(self.E2E_CHUNKS):
            r0, r1 = self.bounds[i], self.bounds[i + 1]
            k0, k1 = int(self.h_ptr[r0]), int(self.h_ptr[r1])
            with torch.cuda.stream(self.copy_s):
                self.q[r0:r1].copy_(hq[r0:r1], non_blocking=True)
                self.indices[k0:k1].copy_(hidx[k0:k1], non_blocking=True)
            cs = comp[i % 2]
            cs.wait_stream(self.copy_s)
            with torch.cuda.stream(cs):
                m.sparse_fwd(self.q[r0:r1], self.rec, self.indptr[r0:r1 + 1], self.indices, c.softmax_scale,
                             has_invalid=True, out=self.out[r0:r1], return_lse=True, lse=self.lse[r0:r1])
            self.d2h_s.wait_stream(cs)
            with torch.cuda.stream(self.d2h_s):
                self.h_out[r0:r1].copy_(self.out[r0:r1], non_blocking=True)
                self.h_lse[r0:r1].copy_(self.lse[r0:r1], non_blocking=True)
        cur.wait_stream(self.comp2_s)
        cur.wait_stream(self.d2h_s)


class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"mla_bench_clocks_{os.getpid()}.csv")
        self.proc = None

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(vals, dist, device):
    """Each value's maximum over the ranks (the slowest rank's time); unchanged on one rank."""
    if dist is None:
        return list(vals)
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(world: int, units_per_rank: float, steps: int, total_ms: float) -> float:
    """Whole-job units per second: every rank processes units_per_rank per step, and the job
    takes the slowest rank's time."""
    return world * units_per_rank * steps / (total_ms * 1e-3)


def capture_step(r, torch):
    """The step's launches captured once into a CUDA graph (replayed per timed step, so that
    the host's per-call marshalling does not leave the GPU idle between the step's kernels);
    None if capture is not possible."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            r.step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            r.step()
        torch.cuda.synchronize()
        return g
    except Exception:
        torch.cuda.synchronize()
        return None


def graph_steps(g, flush, steps, torch):
    """`steps` replays of the captured step, each bracketed by CUDA events, L2 flushed before
    each outside the events.  Returns the step times in ms."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 255)
        ev[i][0].record()
        g.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def timed_steps(r, flush, steps, torch, prof=True):
    """`steps` steps, each bracketed by CUDA events on the current stream (the attention launch
    by the library's profiling hook), L2 flushed before each step outside the events.
    Returns (step times, attention-kernel times) in ms."""
    m = r.m
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ea:      # materialise the handles
        a.record()
        b.record()
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 255)
        if prof:
            m.profile_attention_events(*ea[i])
        ev[i][0].record()
        r.step()
        ev[i][1].record()
    m.profile_attention_events(None, None)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev], [a.elapsed_time(b) for a, b in ea]


def e2e_steps(r, flush, steps, torch):
    """Same steps through the public API with the per-step inputs copied from pinned host
    memory and the results copied back, inside the timed region.  Returns total ms."""
    r.e2e_setup()
    for _ in range(2):
        r.e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total = 0.0
    for i in range(steps):
        flush.fill_(i & 255)
        e0.record()
        r.e2e_step()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    return total


def measure(w: Work, dev, flush, steps: int, warmup: int, min_ms: float, dist, world: int, peak: float,
            peak_kind: str, traffic, cpu_seconds: float):
    """Time one workload: warm-up, then at least `steps` steps and (when min_ms > 0) at least
    min_ms of step time; roofline of its attention kernel, e2e and the oracle baseline."""
    import torch
    r = GpuRunner(w, dev)
    m = r.m
    for _ in range(warmup):
        flush.fill_(1)
        r.step()
    torch.cuda.synchronize()
    assert m.read_device_errors() == 0, f"device error word set during the warm-up of {w.name}"
    K = steps
    if min_ms > 0:
        probe, _ = timed_steps(r, flush, 2, torch, prof=False)
        K = max(steps, int(np.ceil(min_ms / max(min(probe), 1e-3))))
    graph = capture_step(r, torch)
    if graph is not None:
        for _ in range(2):
            graph.replay()
    assert m.read_device_errors() == 0, f"device error word set during the graph capture of {w.name}"
    # the attention kernel's own time: per-launch events of ordinary calls
    _, attn_ms = timed_steps(r, flush, K, torch)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if graph is not None:
        step_ms = graph_steps(graph, flush, K, torch)
    else:
        step_ms, _ = timed_steps(r, flush, K, torch, prof=False)
    total_ms = float(sum(step_ms))
    e2e_ms = e2e_steps(r, flush, K, torch)
    assert m.read_device_errors() == 0, f"device error word set during the timed steps of {w.name}"
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    attn_avg = float(np.mean(attn_ms))
    achieved = w.attn_bytes / (attn_avg * 1e-3) / 1e9
    value = job_rate(world, w.step_bytes, K, total_ms) / 1e9
    res = {
        "steps": K, "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(total_ms / K, 5),
        "query_rows_per_s": round(job_rate(world, w.rows, K, total_ms), 1),
        "row_heads_per_s": round(job_rate(world, w.rows * w.heads, K, total_ms), 1),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": KERNELS[w.name] + " (attention only; epilogue and merge outside)",
                     "kernel_ms": round(attn_avg, 5), "kernel_ms_min": round(float(np.min(attn_ms)), 5),
                     "bytes_per_launch": w.attn_bytes},
        "e2e": {"value": round(job_rate(world, w.step_bytes, K, e2e_ms) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(r.h2d), "d2h_bytes_per_step": int(r.d2h), "mode": r.e2e_mode},
        # tensor-core check: the dense contraction of the launch (rows x heads x visible keys x
        # (2*576 + 2*512) FLOP) over the attention kernel's time, against the bf16 dense peak
        "tensor": {"flops_per_launch": int(w.flops), "achieved_tflops": round(w.flops / (attn_avg * 1e-3) / 1e12, 2),
                   "bf16_peak_tflops": bf16_peak()[0], "frac_of_bf16_peak":
                       round(w.flops / (attn_avg * 1e-3) / 1e12 / bf16_peak()[0], 4), "peak_source": bf16_peak()[1]},
        "gpu_launches": int(r.launches_per_step * K),
        "dtype": w.dtype,
        "config": dict(w.cfg, step_launch="cuda graph replay" if graph is not None else "direct calls"),
    }
    del graph
    del r
    torch.cuda.empty_cache()
    if cpu_seconds > 0:
        res["cpu_baseline"] = cpu_baseline(w, budget_s=cpu_seconds)
    return res


def run_native(args, rank, world, dist):
    import torch
    import mla_latent_cache_attention_gb300 as m
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m.lib()
    peak, peak_kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    full = args.batch == 0 and args.records == 0
    cpu_s = args.cpu_seconds if (rank == 0 and world == 1 and not args.no_cpu_baseline) else 0.0
    w = Work(args.workload, args.batch, args.records)
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    head = measure(w, dev, flush, args.steps, args.warmup, 0.0, dist, world, peak, peak_kind,
                   load_traffic(args.workload) if full else None, 0.0)
    per, works = {}, {}
    if full and not args.headline_only:
        # the other configurations of the path (and the headline past L2), each timed for at
        # least --min-ms so that the clock samples land under load
        for name in [n for n in WORKLOADS if n != args.workload]:
            works[name] = Work(name)
            per[name] = measure(works[name], dev, flush, args.steps, args.warmup, args.min_ms, dist, world, peak,
                                peak_kind, load_traffic(name), 0.0)
        if args.workload == "sparse_prefill":
            name = "sparse_prefill_4M_records"
            works[name] = Work("sparse_prefill", 0, PAST_L2_RECORDS)
            res = measure(works[name], dev, flush, args.steps, args.warmup, args.min_ms, dist, world, peak,
                          peak_kind, load_traffic(name), 0.0)
            res["note"] = ("the headline workload over a 2^22-record pool (2.75 GB, past the 129 MB L2): the "
                           "gathered records come from DRAM")
            per[name] = res
    clocks = clk.stop()
    # the CPU-oracle baselines run after the GPU timing (host work outside every timed region)
    if cpu_s > 0:
        head["cpu_baseline"] = cpu_baseline(w, budget_s=cpu_s)
        for name in per:
            per[name]["cpu_baseline"] = cpu_baseline(works[name], budget_s=max(2.0, cpu_s / 2))
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded numpy)",
        "config": dict(head["config"], l2="flushed between steps (256 MiB write, outside the timed events)",
                       parallelism="replicas" if world > 1 else "single GPU",
                       targets="the three large workloads: sparse prefill (this line), fp8 spec-verify and "
                               "ds_mla H=96 decode (per_config)"),
        "query_rows_per_s": head["query_rows_per_s"], "row_heads_per_s": head["row_heads_per_s"],
        "pct_of_hbm_peak": head["pct_of_hbm_peak"],
        "roofline": head["roofline"], "tensor": head["tensor"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": clocks,
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if per:
        line["per_config"] = per
    return line


def load_traffic(workload):
    """dram bytes per launch of the attention kernel from the committed ncu summary, if any."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            return json.load(f).get(workload)
    except Exception:
        return None


# ------------------------------------------------------------------------------------ CPU oracle arm

def cpu_sample(w: Work, budget_s: float):
    """Time the oracle on a bounded sample of the workload's query rows; returns
    (bytes-equivalent processed per second, rows sampled, seconds)."""
    import oracle
    c = w.case
    rng = np.random.default_rng(0)
    nrows = w.rows

    def run(rows):
        t = time.perf_counter()
        if w.kind == "sparse":
            oracle.sparse_fwd(c.q, c.records, c.indptr, c.indices, c.softmax_scale, True, rows=rows)
        else:
            oracle.paged_decode(c.fmt, c.q, c.cache, c.block_table, c.seq_lens, c.q_len, c.softmax_scale,
                                c.q_scale, c.k_scale, rows=rows)
        return time.perf_counter() - t

    probe = np.sort(rng.choice(nrows, size=min(nrows, 4), replace=False))
    t0 = max(run(probe), 1e-3)
    n = int(max(1, min(nrows, len(probe) * budget_s / t0)))
    rows = np.sort(rng.choice(nrows, size=n, replace=False))
    secs = run(rows)
    frac = (secs, n)
    # the attention bytes of the sampled rows, prorated by rows (q and out) and keys
    if w.kind == "sparse":
        valid = np.zeros(nrows)
        for i, rr in enumerate(rows):
            seg = c.indices[c.indptr[rr]:c.indptr[rr + 1]]
            valid[i] = (seg >= 0).sum()
        b = valid.sum() * 656 + n * w.heads * (576 * 2 + 512 * 2 + 4)
    else:
        eb = w.synth.ENTRY_BYTES[c.fmt]
        qe = 1 if c.fmt == 1 else 2
        # a request's entries are read once for all its q_len rows: charge them per row
        L = c.seq_lens[rows // c.q_len].astype(np.float64)
        b = (L * eb / c.q_len).sum() + n * w.heads * (576 * qe + 512 * 2 + (4 if c.return_lse else 0))
    return b / secs / 1e9, n, secs, frac


def cpu_baseline(w: Work, budget_s: float = 15.0):
    gbs, n, secs, _ = cpu_sample(w, budget_s)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of {w.rows} query rows of {w.name} (all heads), {secs:.1f} s, fp64 C oracle, OpenMP",
            "query_rows_per_s": round(n / secs, 2)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = Work(args.workload, args.batch, args.records)
    budget = max(1.0, args.cpu_seconds / max(1, args.steps))
    vals, rows, secs = [], 0, 0.0
    for _ in range(args.warmup if args.warmup < 1 else 1):
        cpu_sample(w, min(budget, 2.0))
    for _ in range(args.steps):
        gbs, n, s, _ = cpu_sample(w, budget)
        vals.append(gbs)
        rows += n
        secs += s
    value = float(np.mean(vals))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy)", "config": dict(w.cfg),
        "query_rows_per_s": round(rows / secs, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{rows} sampled query rows over {args.steps} steps"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="sparse_prefill", choices=WORKLOADS)
    ap.add_argument("--headline-only", action="store_true",
                    help="time only --workload (no per_config entries); for profiling captures")
    ap.add_argument("--min-ms", type=float, default=250.0,
                    help="GPU time each per_config entry is timed for at least")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests (query rows for sparse_prefill) instead of the workload's own; for small profiling captures")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--records", type=int, default=0,
                    help="sparse_prefill only: size of the record pool (default 65536, L2-resident)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        backend = "nccl" if args.impl == "native" else "gloo"
        dist_mod.init_process_group(backend)
        dist = dist_mod
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_native(args, rank, world, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
