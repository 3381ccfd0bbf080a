"""Benchmark of the MSA hot path on GB300: one JSON line on stdout.

A step is one msa_forward over one batch of the seeded synthetic workload:
the index-key scan with the block max-pool, the top-16 selection and the
attention over the kept blocks.  Default workload: decode batch 4 x 65,536
cached tokens, 4 KV x 16 query heads (value = decode rows/s); a secondary
measurement runs the 4,096-row prompt chunk at an 8,192-token prefix
(prefill rows/s).  Inputs sit in HBM before the timed region.  Where one
step touches more than ~43 MB, the K steps run back to back in one CUDA graph
over 3 to 8 rotating copies of the inputs, so that more than twice the L2 of
other data is read between two uses of a copy (inputs larger than L2); the
one-step time after an L2 flush (a 512 MiB write, then a 256 MiB read so no
dirty line is left; the flush is not timed) is reported beside it, and is
the value for smaller workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle, timed on the host)
Under torchrun each rank runs its own copy of the workload on its own GPU
(decode batches are independent problems: weak scaling, no collective on
the data path); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import platform
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

DECODE_MAX_ROWS = 8  # sequences with up to this many rows take the decode kernels

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILES = os.path.join(ROOT, "profiles")
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


def _peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------- work counts

def _kept_keys(p, top_k=16, S=64):
    J = p // S
    if J + 1 <= top_k:
        return p + 1
    return (top_k - 1) * S + (p % S) + 1


def work_counts(w: synth.Workload):
    """Algorithmic bytes and FLOPs of one step, by stage."""
    H, G, D, Di = w.H, w.G, w.D, w.Di
    dec = [(n, L) for n, L in w.seqs if n <= DECODE_MAX_ROWS]  # decode family: 1 to 8 rows per sequence
    kv_key_bytes_bf16 = D * 2 * 2
    pre = [(n, L) for n, L in w.seqs if n > DECODE_MAX_ROWS]
    # decode scan: every cached index key once (shared by the sequence's rows), the
    # index queries, the pooled scores out
    kh = 1 if w.ik_heads == 1 else H  # index-key heads per position
    scan_bytes = sum(L * kh * Di * 2 + n * H * Di * 2 + n * ((L + 63) // 64) * H * 4 for n, L in dec)
    # decode attention: kept K/V blocks (bf16, or int8 + a 4-byte scale per key for each of
    # K and V), q in, out (fp32) out, per row
    kv_key_bytes = (D * 1 + 4) * 2 if w.kv_dtype == "int8" else D * 2 * 2
    att_bytes = sum(H * (_kept_keys(L - n + i, w.top_k) * kv_key_bytes) + H * G * D * (2 + 4)
                    for n, L in dec for i in range(n))
    # prompt chunks: causal index-score FLOPs and kept-block attention FLOPs
    idx_flops = 0
    att_flops = 0
    for n, L in pre:
        for i in range(n):
            p = L - n + i
            idx_flops += 2 * Di * (p + 1) * H
            att_flops += 4 * D * _kept_keys(p, w.top_k) * H * G
    return dict(scan_bytes=scan_bytes, dec_att_bytes=att_bytes, idx_flops=idx_flops, att_flops=att_flops,
                att_exec_flops=prefill_executed_flops(w), dec_rows=sum(n for n, _ in dec),
                pre_rows=sum(n for n, _ in pre), kv_bytes_frac=kv_key_bytes / kv_key_bytes_bf16)


# Tensor-core FLOPs the prompt-chunk attention issues for one pair of kept
# blocks (128 keys) of one (row, KV head): S^T = K_pair . Q^T (M = 128 keys,
# N = 16 head columns, K = 128 dims) and O^T += V_pair^T . [P_hi; P_lo]^T
# (M = 128 dims, N = 32, K = 128 keys).  Masked keys (past p, the duplicate of
# an odd last block) and the head columns past G are issued too.
EXEC_FLOPS_PER_PAIR = 2 * 128 * 16 * 128 + 2 * 128 * 32 * 128


def prefill_executed_flops(w: synth.Workload):
    """FLOPs the prompt-chunk attention kernel issues on the tensor cores (the
    kept-block FLOPs of work_counts, plus padding and the second P part)."""
    total = 0
    for n, L in w.seqs:
        if n <= DECODE_MAX_ROWS:
            continue
        for i in range(n):
            nsel = min(w.top_k, (L - n + i) // w.S + 1)
            total += (nsel + 1) // 2 * EXEC_FLOPS_PER_PAIR * w.H
    return total


L2_BYTES = 129 << 20


def step_touched_bytes(w: synth.Workload):
    """Bytes one step reads or writes: the decode stages' algorithmic bytes, and
    for prompt chunks q, out (fp32), the index queries and the whole causal
    range of the k, v and index-key caches."""
    wc = work_counts(w)
    b = wc["scan_bytes"] + wc["dec_att_bytes"]
    kh = 1 if w.ik_heads == 1 else w.H
    for n, L in w.seqs:
        if n > DECODE_MAX_ROWS:
            b += n * w.H * w.G * w.D * (2 + 4) + n * w.H * w.Di * 2 + L * (kh * w.Di + 2 * w.H * w.D) * 2
    return b


def rotation_sets(w: synth.Workload, max_sets=8):
    """Input copies for back-to-back timing: enough that the other copies'
    bytes read between two uses of one copy exceed twice the L2; 0 (time with
    an L2 flush before every step instead) when that would take more than
    `max_sets` copies."""
    t = step_touched_bytes(w)
    n = max(3, 1 + -(-2 * L2_BYTES // max(t, 1)))
    return n if n <= max_sets else 0


# ---------------------------------------------------------------- ncu traffic

def _kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_sparse_attention_index_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(summary_name, kernel_files):
    """dram bytes per launch from a committed ncu summary, or None when the
    summary is missing or the kernel source changed since it was taken."""
    path = os.path.join(PROFILES, summary_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != _kernel_source_hash(kernel_files):
        return None
    return int(m.group(1))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            c = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(c[1]))
                mx = float(c[2])
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- ranks

def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the
    value itself when no group is initialised).  `device`: where the
    reduction tensor lives (a CUDA device for NCCL, None/CPU for gloo)."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world_size: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return units_per_rank * world_size / (ms_per_step * 1e-3)


# ---------------------------------------------------------------- the GPU arm

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _to_dev(a, dev):
    """A seeded input on the device: int8 as it is, bf16 bit patterns as bf16."""
    import torch
    if a.dtype == np.int8:
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def measure_gpu(w, steps, warmup, dev, dist_on, flush_bytes=512 << 20, e2e_steps=3, with_e2e=True,
                use_graph=True, page_size=0, rotate_sets=0):
    import torch
    import torch.distributed as td

    import block_sparse_attention_index_gb300 as msa

    x = synth.make_inputs(w)
    scales = {}
    if w.kv_dtype == "int8":  # an int8 key/value cache: its scales go with the problem
        scales = dict(k_scale=torch.from_numpy(x["k_scale"]), v_scale=torch.from_numpy(x["v_scale"]))
    if page_size:  # the same caches as a shuffled page pool with a block table
        pl = synth.paged_layout(w, x, page_size, seed=page_size)
        dx = {k: _to_dev(x[k], dev) for k in ("q", "iq")}
        dx.update({k: _to_dev(pl[k], dev) for k in ("k", "v", "ik")})
        if scales:
            scales = dict(k_scale=torch.from_numpy(pl["k_scale"]), v_scale=torch.from_numpy(pl["v_scale"]))
        pb = msa.Problem(w.H, w.G, w.seqs, dev, top_k=w.top_k, scale=w.softmax_scale,
                         block_table=torch.from_numpy(pl["table"]), page_size=page_size,
                         cache_tokens=pl["num_pages"] * page_size, ik_heads=w.ik_heads, **scales)
        with_e2e = False
    else:
        dx = {k: _to_dev(x[k], dev) for k in ("q", "iq", "k", "v", "ik")}
        pb = msa.Problem(w.H, w.G, w.seqs, dev, top_k=w.top_k, scale=w.softmax_scale, ik_heads=w.ik_heads,
                         **scales)
    ws = pb.workspace()
    out = pb.new_out()
    sel, nsel = pb.new_sel()
    flush = torch.empty(flush_bytes // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(flush_bytes // 8, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(i):
        # write a buffer 4x the L2, then read another 2x the L2 so the lines the
        # write left dirty are written back before the timed step, not during it
        flush.fill_(float(i))
        clean.sum()

    def step(events=None):
        msa.forward(pb, dx["q"], dx["iq"], dx["k"], dx["v"], dx["ik"], out=out, sel=sel, nsel=nsel, workspace=ws,
                    events=events)

    for i in range(warmup):
        flush_l2(i)
        step()
    torch.cuda.synchronize(dev)
    assert msa.error_word(ws) == 0
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for ev in marks:
        ev.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize(dev)
    graph = graph_marked = None
    if use_graph:
        # one step captured once (the library enqueues only its own kernels and event
        # records, never allocates or synchronises) and replayed: no host gaps between
        # the step's kernels.  The timed graph has no marks (a mark between two kernels
        # would break their programmatic-launch overlap); a second graph with marks
        # gives the per-stage times.
        cap = torch.cuda.Stream(dev)
        try:  # mark 0 recorded by torch inside a capture needs an external event
            mark0 = torch.cuda.Event(enable_timing=True, external=True)
            mark0.record(stream)
        except TypeError:
            mark0 = None
        graphs = []
        for ev in (None, marks):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    if ev is not None and mark0 is not None:
                        # stage marks: the flush in the graph, then every mark in line
                        flush_l2(0)
                        mark0.record(cap)
                        step([None] + ev[1:])
                    else:
                        step(ev)
            stream.wait_stream(cap)
            graphs.append(g)
        graph, graph_marked = graphs
        torch.cuda.synchronize(dev)
    # Timed graph: the L2 flush, then the begin mark, the step and the end mark, all
    # captured together (external event-record nodes), so the graph's own launch
    # latency falls before the flush and the timed span holds only the step.
    timed = None
    if use_graph:
        try:
            tmarks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        except TypeError:  # a torch without external events: time around graph.replay()
            tmarks = None
        if tmarks is not None:
            for ev in tmarks:
                ev.record(stream)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    flush_l2(0)
                    # marks in line with the step: an event node on a branch of its
                    # own can fire after the next node of the main branch has run,
                    # so it could start the clock late; in line it can only start it
                    # early (a node-to-node delay before the first kernel)
                    tmarks[0].record(cap)
                    step()
                    tmarks[1].record(cap)
            stream.wait_stream(cap)
            torch.cuda.synchronize(dev)
            for _ in range(warmup):
                g.replay()
            torch.cuda.synchronize(dev)
            timed = g
    begin = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    step_ms, stage_ms = [], []
    if dist_on:
        td.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with ClockSampler(dev.index) as clk:
        if timed is not None:  # one replay per step; its marks are reused, so read them each time
            for i in range(steps):
                timed.replay()
                tmarks[1].synchronize()
                step_ms.append(tmarks[0].elapsed_time(tmarks[1]))
        else:
            for i in range(steps):
                flush_l2(i)
                begin[i].record(stream)
                if graph is not None:
                    graph.replay()
                else:
                    step()
                ends[i].record(stream)
                ends[i].synchronize()
                step_ms.append(begin[i].elapsed_time(ends[i]))
        torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if dist_on:
        td.barrier()
    assert msa.error_word(ws) == 0
    for i in range(steps):  # per-stage times, outside the timed region
        if graph_marked is not None and mark0 is not None:
            graph_marked.replay()  # holds its own flush
            marks[4].synchronize()
            first = [mark0.elapsed_time(marks[1])]
        else:
            flush_l2(i)
            if graph_marked is not None:
                graph_marked.replay()
            else:
                step(marks)
            marks[4].synchronize()
            first = [marks[0].elapsed_time(marks[1])]
        stage_ms.append(first + [marks[j].elapsed_time(marks[j + 1]) for j in range(1, 4)])
    total_ms = max_over_ranks(float(sum(step_ms)), dev if dist_on else None)
    res = dict(ms_per_step=total_ms / steps, stage_ms=np.mean(np.array(stage_ms), axis=0).tolist(),
               wall_s=wall, clocks=clk.summary(), launches=pb.forward_launches() * steps,
               graph=graph is not None, flush_in_graph=timed is not None)

    if rotate_sets > 1 and timed is not None:
        # Steady-state throughput: the K steps back to back in one graph (an L2
        # flush, the begin mark, K msa_forward calls, the end mark), the inputs
        # rotating over `rotate_sets` copies, so every step's inputs were last
        # touched rotate_sets - 1 steps earlier, with more than twice the L2 of
        # other data read in between.  Steps stay serialised on the stream.
        sets = [dx] + [{k: t.clone() for k, t in dx.items()} for _ in range(rotate_sets - 1)]
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                flush_l2(0)
                tmarks[0].record(cap)
                for i in range(steps):
                    d = sets[i % rotate_sets]
                    msa.forward(pb, d["q"], d["iq"], d["k"], d["v"], d["ik"], out=out, sel=sel, nsel=nsel,
                                workspace=ws)
                tmarks[1].record(cap)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        for _ in range(-(-warmup // steps)):  # at least `warmup` untimed steps
            g.replay()
        torch.cuda.synchronize(dev)
        if dist_on:
            td.barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index) as clk2:
            g.replay()
            tmarks[1].synchronize()
            b2b_ms = tmarks[0].elapsed_time(tmarks[1])
            torch.cuda.synchronize(dev)
        if dist_on:
            td.barrier()
        assert msa.error_word(ws) == 0
        res["b2b_ms_per_step"] = max_over_ranks(b2b_ms, dev if dist_on else None) / steps
        res["b2b_sets"] = rotate_sets
        res["b2b_clocks"] = clk2.summary()
        del sets, g
        torch.cuda.synchronize(dev)

    if with_e2e:
        # end to end through the public API from pinned host buffers: every step copies
        # all inputs (q, iq, k, v, ik caches) host->device and reads the output back
        hx = {k: _pinned(x[k]) for k in ("q", "iq", "k", "v", "ik")}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = h_out.numel() * h_out.element_size()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(e2e_steps):
            for k in hx:
                dx[k].copy_(hx[k], non_blocking=True)
            step()
            h_out.copy_(out, non_blocking=True)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        res["e2e_ms"] = ev0.elapsed_time(ev1) / e2e_steps
        res["h2d"], res["d2h"] = h2d, d2h
        if all(n <= DECODE_MAX_ROWS for n, _ in w.seqs) and page_size == 0:
            # resident caches: each step copies only its new inputs (q, iq and the k, v, ik
            # rows of the sequences' new tokens), packed in one pinned staging buffer, in
            # one host->device copy; the rows are scattered into the caches on the device,
            # then the step runs and the output is read back.  The whole sequence is one
            # captured CUDA graph, replayed once per step.
            starts = [int(v) for v in x["cache_starts"]]
            new_idx = [st + L - n + i for st, (n, L) in zip(starts, w.seqs) for i in range(n)]
            idx_h = torch.tensor(new_idx, dtype=torch.long)
            parts = [hx["q"].reshape(-1), hx["iq"].reshape(-1)] + [hx[k][idx_h].reshape(-1) for k in ("k", "v", "ik")]
            sizes = [t.numel() for t in parts]
            h_stage = torch.cat(parts).pin_memory()
            d_stage = torch.empty(h_stage.shape, dtype=h_stage.dtype, device=dev)
            idx_d = idx_h.to(dev)
            views, off = [], 0
            for n_el in sizes:
                views.append(d_stage[off:off + n_el])
                off += n_el

            def e2e_resident_step():
                d_stage.copy_(h_stage, non_blocking=True)
                dx["q"].view(-1).copy_(views[0])
                dx["iq"].view(-1).copy_(views[1])
                for k, v in zip(("k", "v", "ik"), views[2:]):
                    dx[k].index_copy_(0, idx_d, v.view(-1, *dx[k].shape[1:]))
                step()
                h_out.copy_(out, non_blocking=True)

            h2d_r = h_stage.numel() * h_stage.element_size()
            n_res = max(10, steps)
            e2e_resident_step()  # outside any graph first (allocations, warm-up)
            torch.cuda.synchronize(dev)
            g_res = None
            if use_graph:
                g_res = torch.cuda.CUDAGraph()
                cap.wait_stream(stream)
                with torch.cuda.stream(cap):
                    with torch.cuda.graph(g_res, stream=cap):
                        e2e_resident_step()
                stream.wait_stream(cap)
                torch.cuda.synchronize(dev)
                for _ in range(warmup):
                    g_res.replay()
                torch.cuda.synchronize(dev)
            ev0.record(stream)
            for _ in range(n_res):
                if g_res is not None:
                    g_res.replay()
                else:
                    e2e_resident_step()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            assert msa.error_word(ws) == 0
            res["e2e_resident_ms"] = ev0.elapsed_time(ev1) / n_res
            res["h2d_resident"] = h2d_r
            res["e2e_resident_graph"] = g_res is not None
    return res


_ORACLE_INPUTS = {}


def cpu_baseline(w, rows_sample, reps=1, single_thread=True):
    import oracle
    if w.name not in _ORACLE_INPUTS:  # draw the workload once per process
        x = synth.make_inputs(w)
        _ORACLE_INPUTS[w.name] = (x, oracle.Problem.from_workload(w, x))
    x, pr = _ORACLE_INPUTS[w.name]
    threads = oracle.num_threads()
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.forward(pr, x, rows=rows_sample, threads=threads)
    dt = time.perf_counter() - t0
    res = dict(value=len(rows_sample) * reps / dt, unit="rows/s", cores=threads, kind="oracle",
               sample=f"{len(rows_sample)} of {w.total_rows} rows of {w.name}, {reps} rep(s), fp64 C oracle, "
                      f"{threads} OpenMP threads", seconds=dt, cpu_model=_cpu_model())
    if single_thread:  # the same oracle on one core, one row
        one = rows_sample[:1]
        t1 = time.perf_counter()
        oracle.forward(pr, x, rows=one, threads=1)
        res["value_1_thread"] = round(len(one) / (time.perf_counter() - t1), 3)
    return res


def _cpu_model():
    """CPU model of the host (for the oracle baseline), from /proc/cpuinfo."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model", "CPU part"):
        for ln in info:
            if ln.split(":")[0].strip() == key:
                return f"{platform.machine()} {key}: {ln.split(':', 1)[1].strip()}"
    return platform.machine()


def _sample_rows(w, max_rows):
    R = w.total_rows
    if R <= max_rows:
        return list(range(R))
    step = R / max_rows
    return sorted({int(i * step) for i in range(max_rows)})


def _metric_for(w):
    dec = all(n <= DECODE_MAX_ROWS for n, _ in w.seqs)
    pre = all(n > DECODE_MAX_ROWS for n, _ in w.seqs)
    return "MSA decode rows/s" if dec else ("MSA prefill rows/s" if pre else "MSA rows/s (mixed decode + prefill)")


def step_ms(res):
    """The line's time per step: back to back with rotating inputs where that
    was measured, else one step after an L2 flush."""
    return res.get("b2b_ms_per_step", res["ms_per_step"])


def timing_note(res):
    if "b2b_ms_per_step" in res:
        return (f"inputs larger than L2: {res['b2b_sets']} rotating copies of the inputs, steps back to back in one "
                "CUDA graph (an L2 flush, begin mark, K msa_forward calls, end mark)")
    return "flushed before every step (512 MiB write, then 256 MiB read)"


def flushed_latency(res, rows, ws):
    """The one-step figure after an L2 flush, kept beside a back-to-back value."""
    if "b2b_ms_per_step" not in res:
        return None
    return {"value": round(whole_job_rate(rows, ws, res["ms_per_step"]), 1), "unit": "rows/s",
            "ms_per_step": round(res["ms_per_step"], 5),
            "note": "one step per graph replay after an L2 flush, begin and end marks in line"}


def _traffic_source(summary_name, traffic):
    """Where roofline.traffic comes from: a committed ncu capture of the same
    kernel source (not measured in this run), or nothing."""
    if traffic is None:
        return None
    return f"committed ncu capture profiles/{summary_name} (kernel source hash matches); not measured in this run"


def part_work(w, res, hbm, bf16):
    """Each stage's algorithmic work and, where its marked stage time exists,
    its fraction of the measured peak (mixed batches report every part)."""
    wc = work_counts(w)
    st = res["stage_ms"]
    out = {}
    if wc["dec_rows"]:
        out["decode_scan"] = {"bytes": wc["scan_bytes"], "us": round(st[0] * 1e3, 2),
                              "hbm_frac": round(wc["scan_bytes"] / (st[0] * 1e-3) / 1e9 / hbm, 4) if st[0] > 0 else None}
        out["decode_attend"] = {"bytes": wc["dec_att_bytes"], "us": round(st[1] * 1e3, 2),
                                "hbm_frac": round(wc["dec_att_bytes"] / (st[1] * 1e-3) / 1e9 / hbm, 4) if st[1] > 0 else None}
    if wc["pre_rows"]:
        out["prefill_index"] = {"flops": wc["idx_flops"], "us": round(st[2] * 1e3, 2),
                                "bf16_frac": round(wc["idx_flops"] / (st[2] * 1e-3) / 1e12 / bf16, 4) if st[2] > 0 else None}
        out["prefill_attend"] = {"flops": wc["att_flops"], "executed_flops": wc["att_exec_flops"],
                                 "us": round(st[3] * 1e3, 2),
                                 "bf16_frac": round(wc["att_flops"] / (st[3] * 1e-3) / 1e12 / bf16, 4) if st[3] > 0 else None,
                                 "executed_bf16_frac": (round(wc["att_exec_flops"] / (st[3] * 1e-3) / 1e12 / bf16, 4)
                                                        if st[3] > 0 else None)}
    return out


def roofline_for(w, res, hbm, bf16, bf16_sus, peak_kind):
    wc = work_counts(w)
    stage = res["stage_ms"]  # [decode scan, decode attention, prefill index, prefill attention]
    if wc["dec_rows"] and stage[0] > 0:
        achieved = wc["scan_bytes"] / (stage[0] * 1e-3) / 1e9
        traffic = ncu_traffic("decode_scan_4x65536.md", ["decode_scan.cu", "common.cuh"]) if w.name == "decode_4x65536" else None
        return {"kernel": "decode_scan_kernel", "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                "traffic_source": _traffic_source("decode_scan_4x65536.md", traffic),
                "algorithmic_bytes": wc["scan_bytes"], "kernel_us": round(stage[0] * 1e3, 2),
                "peak_source": f"{peak_kind} hbm_gbs (copy)"}
    if stage[3] > 0:
        achieved = wc["att_flops"] / (stage[3] * 1e-3) / 1e12
        traffic = (ncu_traffic("prefill_attend_4096_at_8192.md", ["prefill_attend.cu", "common.cuh"])
                   if w.name == "prefill_4096_at_8192" else None)
        executed = wc["att_exec_flops"] / (stage[3] * 1e-3) / 1e12
        # the indexer's FLOPs counted with the attention's, over both stages (the second figure the
        # prompt-chunk target is stated for)
        both = ((wc["att_flops"] + wc["idx_flops"]) / ((stage[2] + stage[3]) * 1e-3) / 1e12
                if stage[2] > 0 else None)
        return {"kernel": "prefill_attend_kernel", "bound": "tensor", "achieved": round(achieved, 1), "peak": bf16,
                "unit": "TFLOP/s", "frac": round(achieved / bf16, 4), "traffic": traffic,
                "traffic_source": _traffic_source("prefill_attend_4096_at_8192.md", traffic),
                "algorithmic_flops": wc["att_flops"], "executed_flops": wc["att_exec_flops"],
                "executed_tflops": round(executed, 1), "executed_frac": round(executed / bf16, 4),
                "with_indexer_flops": wc["att_flops"] + wc["idx_flops"],
                "with_indexer_frac": round(both / bf16, 4) if both is not None else None,
                "kernel_us": round(stage[3] * 1e3, 2), "peak_source": f"{peak_kind} bf16_tflops (burst)"}
    return None


def l2_note(w, use_graph=True):
    """How the L2 is kept out of the timing for workload w (the rule this
    bench applies to it; the same words in both arms' config)."""
    sets = rotation_sets(w)
    if sets > 1 and use_graph:
        return (f"inputs larger than L2: {sets} rotating copies of the inputs, steps back to back in one CUDA graph "
                "(an L2 flush, begin mark, K msa_forward calls, end mark)")
    return "flushed before every step (512 MiB write, then 256 MiB read)"


def config_for(w, world_size, use_graph=True):
    """The workload description printed by both arms (identical dicts)."""
    return {"workload": w.name, "note": w.note, "H": w.H, "G": w.G, "head_dim": w.D, "index_dim": w.Di,
            "block": w.S, "top_k": w.top_k, "rows_per_gpu": w.total_rows, "cache_tokens_per_gpu": w.cache_tokens,
            "l2": l2_note(w, use_graph), "parallelism": f"replicas x{world_size}"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_4x65536", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--secondary", default="prefill_4096_at_8192",
                    help="second workload measured in the same run ('none' to skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each step directly instead of replaying a CUDA graph")
    ap.add_argument("--multirow", default="decode_4x4_65536",
                    help="decode workload with several rows per sequence measured in the same run ('none' to skip)")
    ap.add_argument("--no-other-configs", dest="other_configs", action="store_false",
                    help="skip the short timings of the remaining configurations")
    ap.add_argument("--shared-key", default="decode_4x65536_shared_ik",
                    help="decode workload with one index key shared by all KV heads ('none' to skip)")
    ap.add_argument("--int8", default="decode_4x65536_int8",
                    help="decode workload with an int8 key/value cache measured in the same run ('none' to skip)")
    ap.add_argument("--int8-prefill", default="prefill_4096_at_8192_int8",
                    help="prompt-chunk workload with an int8 key/value cache measured in the same run ('none' to skip)")
    ap.add_argument("--paged-page-size", type=int, default=64,
                    help="also time the primary workload from a paged cache with this page size (0: skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = _dist()
    w = synth.workload(args.workload)
    hbm, bf16, bf16_sus, peak_kind = _peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        steps_done, t_total = 0, 0.0
        rows = _sample_rows(w, 4 if all(n <= DECODE_MAX_ROWS for n, _ in w.seqs) else 64)
        for i in range(args.warmup + args.steps):
            r = cpu_baseline(w, rows, single_thread=False)
            if i >= args.warmup:
                steps_done += 1
                t_total += r["seconds"]
        value = len(rows) * steps_done / t_total
        line = {"impl": "reference", "metric": _metric_for(w), "value": value, "unit": "rows/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * t_total / steps_done, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_for(w, ws, use_graph=not args.no_graph),
                "cpu_baseline": {"kind": "oracle", "cores": r["cores"], "sample": r["sample"], "value": value,
                                 "unit": "rows/s", "sample_rows": len(rows)},
                "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import torch.distributed as td
    dist_on = ws > 1
    if dist_on:
        td.init_process_group("nccl")
    dev = torch.device("cuda", local if dist_on else 0)
    torch.cuda.set_device(dev)

    res = measure_gpu(w, args.steps, args.warmup, dev, dist_on, with_e2e=not args.no_e2e,
                      use_graph=not args.no_graph, rotate_sets=rotation_sets(w))
    rows = w.total_rows
    value = whole_job_rate(rows, ws, step_ms(res))
    line = {"metric": _metric_for(w), "value": round(value, 1), "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms(res), 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_for(w, ws, use_graph=not args.no_graph),
            "l2": timing_note(res),
            "launch": ("CUDA graph: L2 flush, begin mark, one msa_forward, end mark (marks in line)"
                       if res.get("flush_in_graph") and "b2b_ms_per_step" not in res
                       else "CUDA graph: L2 flush, begin mark, K msa_forward calls, end mark"
                       if "b2b_ms_per_step" in res
                       else "CUDA graph replay of one msa_forward" if res["graph"] else "direct msa_forward calls"),
            "stage_us": {"decode_scan": round(res["stage_ms"][0] * 1e3, 2),
                         "decode_attend": round(res["stage_ms"][1] * 1e3, 2),
                         "prefill_index": round(res["stage_ms"][2] * 1e3, 2),
                         "prefill_attend": round(res["stage_ms"][3] * 1e3, 2)},
            "roofline": roofline_for(w, res, hbm, bf16, bf16_sus, peak_kind),
            "clocks": res.get("b2b_clocks", res["clocks"]), "gpu_launches": res["launches"]}
    if flushed_latency(res, rows, ws):
        line["latency_flushed"] = flushed_latency(res, rows, ws)
    wc = work_counts(w)
    step_bytes = wc["scan_bytes"] + wc["dec_att_bytes"]
    if step_bytes and wc["pre_rows"] == 0:
        line["step_hbm_frac"] = round(step_bytes / (step_ms(res) * 1e-3) / 1e9 / hbm, 4)
    if "e2e_ms" in res:
        line["e2e"] = {"value": round(whole_job_rate(rows, ws, max_over_ranks(res["e2e_ms"], dev if dist_on else None)), 1),
                       "unit": "rows/s",
                       "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                       "note": "every step copies q, iq and the k, v, ik caches from pinned host memory and reads "
                               "the output back"}
    if "e2e_resident_ms" in res:
        line["e2e_resident_cache"] = {
            "value": round(whole_job_rate(rows, ws, max_over_ranks(res["e2e_resident_ms"], dev if dist_on else None)), 1),
            "unit": "rows/s", "h2d_bytes_per_step": res["h2d_resident"], "d2h_bytes_per_step": res["d2h"],
            "note": "caches resident on the GPU; every step copies q, iq and the new tokens' k, v, ik rows from "
                    "one pinned host buffer, scatters the rows into the caches, runs msa_forward and reads the "
                    "output back" + (", all in one CUDA graph replayed per step" if res.get("e2e_resident_graph")
                                     else "") + " (the full-cache copy of e2e is bound by the host link, ~210 GB/s)"}
    if args.secondary != "none" and args.secondary != args.workload:
        w2 = synth.workload(args.secondary)
        res2 = measure_gpu(w2, max(3, args.steps // 2), args.warmup, dev, dist_on, with_e2e=False,
                           use_graph=not args.no_graph, rotate_sets=rotation_sets(w2))
        line["secondary"] = {"metric": _metric_for(w2), "workload": w2.name,
                             "value": round(whole_job_rate(w2.total_rows, ws, step_ms(res2)), 1), "unit": "rows/s",
                             "ms_per_step": round(step_ms(res2), 5), "l2": timing_note(res2),
                             "latency_flushed": flushed_latency(res2, w2.total_rows, ws),
                             "stage_us": {"prefill_index": round(res2["stage_ms"][2] * 1e3, 2),
                                          "prefill_attend": round(res2["stage_ms"][3] * 1e3, 2)},
                             "roofline": roofline_for(w2, res2, hbm, bf16, bf16_sus, peak_kind),
                             "parts": part_work(w2, res2, hbm, bf16), "gpu_launches": res2["launches"]}
        line["gpu_launches"] += res2["launches"]
    if args.paged_page_size > 0:
        resp = measure_gpu(w, args.steps, args.warmup, dev, dist_on, with_e2e=False, use_graph=not args.no_graph,
                           page_size=args.paged_page_size, rotate_sets=rotation_sets(w))
        line["paged"] = {"page_size": args.paged_page_size, "workload": w.name,
                         "value": round(whole_job_rate(rows, ws, step_ms(resp)), 1),
                         "unit": "rows/s", "ms_per_step": round(step_ms(resp), 5), "l2": timing_note(resp),
                         "latency_flushed": flushed_latency(resp, rows, ws),
                         "note": "same inputs from a shuffled page pool addressed through a block table"}
        line["gpu_launches"] += resp["launches"]
    for key, name in (("shared_key", args.shared_key), ("int8", args.int8), ("int8_prefill", args.int8_prefill)):
        if name == "none" or name == args.workload:
            continue
        w4 = synth.workload(name)
        res4 = measure_gpu(w4, args.steps, args.warmup, dev, dist_on, with_e2e=False, use_graph=not args.no_graph,
                           rotate_sets=rotation_sets(w4))
        line[key] = {"metric": _metric_for(w4), "workload": w4.name,
                     "value": round(whole_job_rate(w4.total_rows, ws, step_ms(res4)), 1),
                     "unit": "rows/s", "ms_per_step": round(step_ms(res4), 5), "l2": timing_note(res4),
                     "latency_flushed": flushed_latency(res4, w4.total_rows, ws),
                     "stage_us": {k: round(v * 1e3, 2) for k, v in zip(
                         ("decode_scan", "decode_attend", "prefill_index", "prefill_attend"), res4["stage_ms"])},
                     "roofline": roofline_for(w4, res4, hbm, bf16, bf16_sus, peak_kind), "note": w4.note,
                     "kv_bytes_frac_of_bf16": round(work_counts(w4)["kv_bytes_frac"], 4)}
        line["gpu_launches"] += res4["launches"]
    if args.multirow != "none" and args.multirow != args.workload:
        w3 = synth.workload(args.multirow)
        res3 = measure_gpu(w3, args.steps, args.warmup, dev, dist_on, with_e2e=False, use_graph=not args.no_graph,
                           rotate_sets=rotation_sets(w3))
        line["multirow"] = {"metric": _metric_for(w3), "workload": w3.name,
                            "value": round(whole_job_rate(w3.total_rows, ws, step_ms(res3)), 1),
                            "unit": "rows/s", "ms_per_step": round(step_ms(res3), 5), "l2": timing_note(res3),
                            "latency_flushed": flushed_latency(res3, w3.total_rows, ws),
                            "stage_us": {"decode_scan": round(res3["stage_ms"][0] * 1e3, 2),
                                         "decode_attend": round(res3["stage_ms"][1] * 1e3, 2)},
                            "roofline": roofline_for(w3, res3, hbm, bf16, bf16_sus, peak_kind),
                            "note": w3.note}
        line["gpu_launches"] += res3["launches"]
    if args.other_configs:
        # the remaining configurations of the pages' workloads, a short timing each
        others = []
        for name in ("decode_1x4096", "decode_1x262144", "mixed_8dec_512pre"):
            if name in (args.workload, args.secondary):
                continue
            w5 = synth.workload(name)
            res5 = measure_gpu(w5, max(5, args.steps // 2), args.warmup, dev, dist_on, with_e2e=False,
                               use_graph=not args.no_graph, rotate_sets=rotation_sets(w5))
            rf = roofline_for(w5, res5, hbm, bf16, bf16_sus, peak_kind)
            wc5 = work_counts(w5)
            sb = wc5["scan_bytes"] + wc5["dec_att_bytes"]
            others.append({"workload": w5.name, "metric": _metric_for(w5),
                           "value": round(whole_job_rate(w5.total_rows, ws, step_ms(res5)), 1), "unit": "rows/s",
                           "ms_per_step": round(step_ms(res5), 5), "l2": timing_note(res5),
                           "latency_flushed": flushed_latency(res5, w5.total_rows, ws),
                           "stage_us": {k: round(v * 1e3, 2) for k, v in zip(
                               ("decode_scan", "decode_attend", "prefill_index", "prefill_attend"), res5["stage_ms"])},
                           "roofline": rf, "parts": part_work(w5, res5, hbm, bf16),
                           "decode_step_hbm_frac": (round(sb / (step_ms(res5) * 1e-3) / 1e9 / hbm, 4)
                                                    if wc5["pre_rows"] == 0 and sb else None)})
            line["gpu_launches"] += res5["launches"]
        line["other_configs"] = others
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline(w, _sample_rows(w, 4 if wc["pre_rows"] == 0 else 64), reps=3 if wc["pre_rows"] == 0 else 1)
        cb.pop("seconds")
        line["cpu_baseline"] = cb
    if dist_on:
        td.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
