#!/usr/bin/env python
"""Benchmark of the GB300 GQA attention library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--paths all|main]

Prints ONE JSON line on rank 0.  The headline is the causal prefill at
head_dim 256 (2048 queries over 2048 keys, 16 query / 8 KV heads, f16 K/V,
scale 1): `value` is algorithmic TFLOP/s (4*d FLOPs per visible
(query, key) pair and head) over the device time of one call through the C
ABI with inputs resident in HBM.  `paths` adds, measured in the same run,
the head_dim-512 prefix prefill (TFLOP/s), the paged decode (KV GB/s) and
the speculative-verify chain pack -> mask -> attention -> commit (GB/s of
algorithmic bytes).  Every input is seeded and synthetic (workloads module).

Timing: W untimed warm-up steps, then K steps, each preceded by an L2 flush
(a 512 MiB device write, outside the step's CUDA-event pair) and timed with
CUDA events on the launching stream, bracketed by a barrier and a device
synchronisation.  `roofline` times the dominant kernel alone with events the
library records around its launch (gqa_timing_enable).  SM clocks are sampled
with nvidia-smi during the timed region.  Under torchrun (N>1) every rank runs
an independent replica (the path shards into independent problems; no
collective is on the data path) and the slowest rank's time is used.

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload on the host cores (the only implementation the pages allow to
run here).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import pathlib
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "prefill attn TFLOP/s & decode/verify KV GB/s (1×GB300, % of roofline)"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------
def peaks() -> tuple[dict, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return d, "measured"
        except Exception:
            pass
    return FALLBACK, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict | None:
        if self.proc is None or not self.path:
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "reasons": reasons}


def traffic_for(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source has changed since the counters were taken."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    try:
        table = json.loads(p.read_text())
    except Exception:
        return None
    e = table.get(f"{kernel}@{workload}")
    if not e:
        return None
    src = ROOT / e["source"]
    if not src.exists() or hashlib.sha256(src.read_bytes()).hexdigest() != e["source_sha256"]:
        return None
    return float(e["bytes_per_launch"])


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
class Timer:
    def __init__(self, torch, dist):
        self.torch = torch
        self.dist = dist
        self.flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        self.graphs_used = False

    def flush(self):
        self.flush_buf.zero_()

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def graph(self, fn):
        """fn captured into a CUDA graph (after the caller's eager warm-up): replaying it
        submits the step's launches at once, so host-side launch overhead (ctypes
        marshalling, argument checks) stays off the device timeline.  Falls back to
        fn itself if the step cannot be captured."""
        torch = self.torch
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                fn()
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            torch.cuda.synchronize()
            self.graphs_used = True
            return g.replay
        except Exception as e:  # noqa: BLE001 -- report and time eagerly
            print(f"graph capture failed ({e}); timing eagerly", file=sys.stderr)
            torch.cuda.synchronize()
            self.graphs_used = False
            return fn

    def steps(self, fn, steps: int, warmup: int, graph: bool = True) -> list[float]:
        """Per-step device ms of fn (L2 flushed before each step), replayed as a CUDA
        graph unless graph=False."""
        torch = self.torch
        for _ in range(warmup):
            self.flush()
            fn()
        self.barrier()
        if graph:
            fn = self.graph(fn)
            for _ in range(2):
                self.flush()
                fn()
            self.barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            self.flush()
            e0.record()
            fn()
            e1.record()
        self.barrier()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    def kernel_ms(self, g, fn, reps: int) -> float:
        """Mean device ms of the dominant kernel of fn's last library call: the
        library records CUDA events around that launch (event nodes of the graph)."""
        g.gqa_timing_enable(True)
        out = []
        try:
            fn = self.graph(fn)
            for _ in range(reps):
                self.flush()
                fn()
                out.append(g.gqa_timing_last_ms())
        finally:
            g.gqa_timing_enable(False)
        return sum(out) / len(out)

    def max_over_ranks(self, x: float) -> float:
        return max_over_ranks(self.torch, self.dist, x)


def max_over_ranks(torch, dist, x: float) -> float:
    """The slowest rank's value (every rank gets it); x itself without a process group.
    The reduction runs on the device the group's backend serves (CUDA for NCCL)."""
    if dist is None:
        return x
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workloads: each returns (step_fn, info) with algorithmic work per step
# ---------------------------------------------------------------------------
def _dev(torch, a, kind=None):
    a = np.ascontiguousarray(a)
    if kind == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    if kind == "u32":
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(a).cuda()


class E2EPipe:
    """End-to-end prefill steps double-buffered over three streams: step i's inputs go
    host -> device on one stream while step i-1's attention runs on a second and its
    output goes device -> host on a third.  Every step still copies its own inputs in
    from pinned host memory and its result out; buffer set i % 2 is reused only after
    the attention and the read-back of step i-2 that used it are done."""

    def __init__(self, torch, g, case, host_in, dev0):
        self.torch, self.g, self.case = torch, g, case
        self.host_in = host_in
        self.sets = [dev0, tuple(torch.empty_like(t) for t in dev0)]
        self.hout = [torch.empty(dev0[4].shape, dtype=torch.float32).pin_memory()
                     for _ in range(2)]
        self.s_in, self.s_cmp, self.s_out = (torch.cuda.Stream() for _ in range(3))
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_in, self.ev_kern, self.ev_out = ev(), ev(), ev()
        self.used = [False, False]

    def step(self, i: int):
        torch, b = self.torch, i % 2
        q, k, v, m, out, ws = self.sets[b]
        with torch.cuda.stream(self.s_in):
            if self.used[b]:
                self.s_in.wait_event(self.ev_kern[b])
            for d, h in zip((q, k, v, m), self.host_in):
                d.copy_(h, non_blocking=True)
            self.ev_in[b].record()
        with torch.cuda.stream(self.s_cmp):
            self.s_cmp.wait_event(self.ev_in[b])
            if self.used[b]:
                self.s_cmp.wait_event(self.ev_out[b])
            self.g.gqa_attn_prefill(q, k, v, m, self.case.scale, out=out, workspace=ws)
            self.ev_kern[b].record()
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_kern[b])
            self.hout[b].copy_(out, non_blocking=True)
            self.ev_out[b].record()
        self.used[b] = True

    def run(self, steps: int, warmup: int) -> float:
        """Mean device ms per step over `steps` pipelined steps, after `warmup` of them;
        CUDA events on the current stream bracket the run, joined to all three streams."""
        torch = self.torch
        cur = torch.cuda.current_stream()
        for i in range(warmup):
            self.step(i)
        for s in (self.s_in, self.s_cmp, self.s_out):
            cur.wait_stream(s)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for s in (self.s_in, self.s_cmp, self.s_out):
            s.wait_stream(cur)
        for i in range(warmup, warmup + steps):
            self.step(i)
        for s in (self.s_in, self.s_cmp, self.s_out):
            cur.wait_stream(s)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps


def host_io(torch, step, inputs, outputs):
    """The same step end to end: every call first copies `inputs` (device tensors) in
    from pinned host copies made here, then runs `step`, then reads `outputs` back into
    pinned host memory.  Returns (e2e step, h2d bytes, d2h bytes)."""
    hin = [t.cpu().pin_memory() for t in inputs]
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outputs]

    def e2e_step():
        for d, h in zip(inputs, hin):
            d.copy_(h, non_blocking=True)
        step()
        for h, d in zip(hout, outputs):
            h.copy_(d, non_blocking=True)

    nb = lambda t: t.numel() * t.element_size()
    return e2e_step, sum(nb(t) for t in inputs), sum(nb(t) for t in outputs)


def setup_prefill(torch, g, case):
    kind = "bf16" if case.kv_dtype == "bf16" else None
    q, k, v, m = (_dev(torch, case.q), _dev(torch, case.k, kind), _dev(torch, case.v, kind),
                  _dev(torch, case.mask))
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, g.gqa_attn_prefill_workspace_size(case.rows, case.n_heads,
                                                              case.n_kv_heads, case.head_dim,
                                                              case.kv_pad)),
                     dtype=torch.uint8, device="cuda")

    def step():
        g.gqa_attn_prefill(q, k, v, m, case.scale, out=out, workspace=ws)

    # host copies of the same inputs for the end-to-end measurement
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, hm = pin(q), pin(k), pin(v), pin(m)
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        m.copy_(hm, non_blocking=True)
        g.gqa_attn_prefill(q, k, v, m, case.scale, out=out, workspace=ws)
        hout.copy_(out, non_blocking=True)

    e2e_step.pipe = lambda: E2EPipe(torch, g, case, (hq, hk, hv, hm), (q, k, v, m, out, ws))

    nb = lambda t: t.numel() * t.element_size()
    # classification pre-pass + attention kernel (these workloads need no key split)
    info = {"flops": case.flops(), "h2d": nb(q) + nb(k) + nb(v) + nb(m), "d2h": nb(out),
            "launches": 2}
    return step, e2e_step, info


def setup_decode(torch, g, c):
    q, kp, vp = _dev(torch, c.q), _dev(torch, c.k_pool), _dev(torch, c.v_pool)
    pt, cl = _dev(torch, c.page_table), _dev(torch, c.context_lens)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(g.gqa_attn_paged_decode_workspace_size(c.num_seqs, c.n_heads, c.head_dim,
                                                            c.max_pages_per_seq, c.page_size),
                     dtype=torch.uint8, device="cuda")

    def step():
        g.gqa_attn_paged_decode(q, kp, vp, pt, cl, c.scale, out=out, workspace=ws)

    pages_used = int(sum(-(-int(x) // c.page_size) for x in c.context_lens))
    kv = c.kv_bytes()
    qo = q.numel() * 4
    info = {"bytes": kv + 2 * qo + pages_used * 4 + c.num_seqs * 4,
            "kernel_bytes": kv + qo + pages_used * 4 + c.num_seqs * 4, "kv_bytes": kv,
            "launches": 2}
    # end to end: the step's queries, page table and context lengths in, O out (the KV
    # pools are the resident cache, not a per-step input)
    info["e2e"] = host_io(torch, step, [q, pt, cl], [out])
    return step, info


def setup_verify(torch, g, c):
    B, H, HK, D, R, W, K, MC = c.geom
    rk, rv = _dev(torch, c.ring_k, "bf16"), _dev(torch, c.ring_v, "bf16")
    cq, ck, cv = _dev(torch, c.cur_q), _dev(torch, c.cur_k), _dev(torch, c.cur_v)
    nk, nv = _dev(torch, c.new_k), _dev(torch, c.new_v)
    lens, pos = _dev(torch, c.cache_lengths, "u32"), _dev(torch, c.write_positions, "u32")
    cnt = _dev(torch, c.commit_counts, "u32")
    pq = torch.empty((B, H, R, D), dtype=torch.bfloat16, device="cuda")
    pk = torch.empty((B, HK, K, D), dtype=torch.bfloat16, device="cuda")
    pv = torch.empty_like(pk)
    mask = torch.empty((B, H, R, K), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, R, H, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, g.gqa_attn_verify_workspace_size(c.geom)), dtype=torch.uint8,
                     device="cuda")
    ops = {
        "pack": lambda: g.gqa_pack_attention(rk, rv, cq, ck, cv, lens, pos, pq, pk, pv, c.geom),
        "mask": lambda: g.gqa_fill_mask(lens, mask, c.geom),
        "attn": lambda: g.gqa_attn_verify(pq, pk, pv, mask, c.geom, c.scale, out=out,
                                          workspace=ws),
        "commit": lambda: g.gqa_commit_kv(nk, nv, cnt, pos, rk, rv, c.geom),
    }

    def step():
        for f in ops.values():
            f()

    fused_out = torch.empty((B, R, H, D), dtype=torch.float32, device="cuda")
    fws = torch.empty(max(1, g.gqa_attn_verify_ring_workspace_size(c.geom)), dtype=torch.uint8,
                      device="cuda")
    fused = {
        "attn": lambda: g.gqa_attn_verify_ring(rk, rv, cq, ck, cv, lens, pos, c.geom, c.scale,
                                               out=fused_out, workspace=fws),
        "commit": ops["commit"],
    }
    hist = int(sum(min(int(x), W - 1) for x in c.cache_lengths))
    n_commit = int(sum(min(int(x), MC) for x in c.commit_counts))
    nb = lambda t: t.numel() * t.element_size()
    by = {
        "pack": hist * HK * D * 2 * 2 + nb(cq) + nb(ck) + nb(cv) + nb(pq) + nb(pk) + nb(pv),
        "mask": nb(mask),
        "attn": nb(pq) + nb(pk) + nb(pv) + nb(mask) + nb(out),
        "commit": n_commit * HK * D * (4 + 2) * 2,
    }
    # fused: the visible history once, the current rows, O
    fby = {"attn": hist * HK * D * 2 * 2 + nb(cq) + nb(ck) + nb(cv) + nb(out),
           "commit": by["commit"]}
    # end to end: the draft rows (current Q/K/V, the rows to commit) and the lanes'
    # counters in, O out (the rings are the resident cache)
    step_in = [cq, ck, cv, nk, nv, lens, pos, cnt]

    def fstep():
        for f in fused.values():
            f()

    return step, ops, {"bytes": by, "launches": 1 + 1 + 2 + 1, "fused": fused,
                       "fused_bytes": fby, "fused_launches": 1 + 1 + 1,
                       "e2e": host_io(torch, step, step_in, [out]),
                       "fused_e2e": host_io(torch, fstep, step_in, [fused_out])}


def setup_chunk(torch, g, c):
    """Chunked prefill over pages: append the new tokens' K/V into their pages, then
    attend (each new token over its sequence's cached prefix and the new tokens up to
    itself)."""
    q, kn, vn = _dev(torch, c.q), _dev(torch, c.k_new), _dev(torch, c.v_new)
    kp, vp = _dev(torch, c.k_pool), _dev(torch, c.v_pool)
    pt, off, ps = _dev(torch, c.page_table), _dev(torch, c.token_offsets), _dev(torch, c.position_start)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    max_tok = int(np.diff(c.token_offsets).max())
    ws = torch.empty(max(1, g.gqa_attn_paged_prefill_workspace_size(
        c.num_seqs, max_tok, c.n_heads, c.n_kv_heads, c.head_dim, c.max_pages_per_seq,
        c.page_size)), dtype=torch.uint8, device="cuda")
    ops = {
        "append": lambda: g.gqa_paged_append(kn, vn, off, ps, pt, kp, vp),
        "attn": lambda: g.gqa_attn_paged_prefill(q, kp, vp, pt, off, ps, max_tok, c.scale,
                                                 out=out, workspace=ws),
    }

    def step():
        for f in ops.values():
            f()

    nb = lambda t: t.numel() * t.element_size()
    # append: f32 rows in, 16-bit rows out, for K and V
    append_bytes = nb(kn) + nb(vn) + (nb(kn) + nb(vn)) // 2
    # append, unit ordering, attention
    # end to end: the new tokens' Q, K and V, the offsets, start positions and page table
    # in, O out (the page pools are the resident cache)
    return step, ops, {"flops": c.flops(), "append_bytes": append_bytes, "launches": 3,
                       "e2e": host_io(torch, step, [q, kn, vn, off, ps, pt], [out])}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_prefill_sample(case, n_pairs: int, seed: int = 0):
    """Time the float64 oracle on n_pairs sampled (row, head) outputs; returns
    (seconds, algorithmic flops of the sample)."""
    import oracle
    rng = np.random.default_rng(seed)
    pairs = np.stack([rng.integers(0, case.rows, n_pairs), rng.integers(0, case.n_heads, n_pairs)],
                     axis=1).astype(np.int32)
    vis = (case.mask == 0).sum(axis=1)
    flops = float(4.0 * case.head_dim * vis[pairs[:, 0]].sum())
    t0 = time.perf_counter()
    oracle.attention(case.q, case.k, case.v, kv_dtype=case.kv_dtype, scale=case.scale,
                     mask=case.mask, pairs=pairs)
    return time.perf_counter() - t0, flops


def cpu_baseline(case, target_s: float = 12.0) -> dict:
    import oracle
    t, f = oracle_prefill_sample(case, 64)
    per_pair = max(t / 64, 1e-6)
    n = int(min(case.rows * case.n_heads, max(64, target_s / per_pair)))
    t, f = oracle_prefill_sample(case, n, seed=1)
    return {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} random (query row, head) outputs of {case.name} "
                      f"({f / 1e9:.1f} GFLOP, {t:.1f} s), float64 C with OpenMP"}


def _cpu_line(value: float, unit: str, sample: str) -> dict:
    import oracle
    return {"value": value, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample}


def cpu_prefill(case, target_s: float = 3.0) -> dict:
    """The oracle on sampled (query row, head) outputs of a prefill workload."""
    t, _ = oracle_prefill_sample(case, 16)
    n = int(min(case.rows * case.n_heads, max(16, target_s / max(t / 16, 1e-6))))
    t, f = oracle_prefill_sample(case, n, seed=2)
    return _cpu_line(f / t / 1e12, "TFLOP/s",
                     f"{n} random (query row, head) outputs ({f / 1e9:.1f} GFLOP, {t:.1f} s)")


def cpu_decode(c, target_s: float = 3.0) -> dict:
    """The oracle's paged decode of a random subset of the sequences; GB/s of their K/V."""
    import oracle
    order = np.random.default_rng(3).permutation(c.num_seqs).astype(np.int32)
    per_tok = c.n_kv_heads * c.head_dim * 2 * 2

    def run(seqs):
        t0 = time.perf_counter()
        oracle.paged_decode(c.q, c.k_pool, c.v_pool, kv_dtype=c.kv_dtype, page_table=c.page_table,
                            context_lens=c.context_lens, scale=c.scale, seqs=seqs)
        return time.perf_counter() - t0, int(c.context_lens[seqs].astype(np.int64).sum()) * per_tok

    t, b = run(order[:1])
    budget = b / max(t, 1e-6) * target_s  # bytes the oracle gets through in target_s
    lens = c.context_lens[order].astype(np.int64) * per_tok
    n = int(min(c.num_seqs, max(1, np.searchsorted(np.cumsum(lens), budget) + 1)))
    t, b = run(order[:n])
    return _cpu_line(b / t / 1e9, "GB/s",
                     f"{n} of {c.num_seqs} sequences ({b / 1e9:.2f} GB of K/V, {t:.1f} s)")


def cpu_verify(c, chain_bytes: int, fused_bytes: int) -> tuple[dict, dict]:
    """The oracle's verify step on the whole workload: pack, mask, attention over the
    packed copy and commit; and the attention read straight from the ring."""
    import oracle
    t0 = time.perf_counter()
    pq, pk, pv = oracle.pack_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v,
                                       c.cache_lengths, c.write_positions, c.geom)
    m = oracle.fill_mask(c.cache_lengths, c.geom)
    oracle.verify_attention(pq, pk, pv, m, c.geom, c.scale)
    oracle.commit_kv(c.new_k, c.new_v, c.commit_counts, c.write_positions, c.ring_k, c.ring_v, c.geom)
    t_chain = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.verify_ring_attention(c.ring_k, c.ring_v, c.cur_q, c.cur_k, c.cur_v, c.cache_lengths,
                                 c.write_positions, c.geom, c.scale)
    oracle.commit_kv(c.new_k, c.new_v, c.commit_counts, c.write_positions, c.ring_k, c.ring_v, c.geom)
    t_fused = time.perf_counter() - t0
    return (_cpu_line(chain_bytes / t_chain / 1e9, "GB/s", f"the whole step ({t_chain:.2f} s)"),
            _cpu_line(fused_bytes / t_fused / 1e9, "GB/s", f"the whole step ({t_fused:.2f} s)"))


def cpu_chunk(c, target_s: float = 3.0) -> dict:
    """The oracle's page append and chunked prefill for the first tokens of one sequence
    (the one with the longest cached prefix)."""
    import oracle
    counts = np.diff(c.token_offsets)
    s = int(np.argmax(np.where(counts > 0, c.position_start, -1)))
    o0, ps = int(c.token_offsets[s]), int(c.position_start[s])
    ntok = int(c.token_offsets[s + 1]) - o0
    strides = dict(page_stride=c.k_pool.strides[0] // 2, token_stride=c.k_pool.strides[1] // 2,
                   head_stride=c.k_pool.strides[2] // 2)

    def run(n):
        offs = np.array([0, n], np.int32)
        pos = np.array([ps], np.int32)
        pt = c.page_table[s:s + 1]
        t0 = time.perf_counter()
        kp, vp, _ = oracle.paged_append(c.k_new[o0:o0 + n], c.v_new[o0:o0 + n], offs, pos, pt,
                                        c.k_pool, c.v_pool, kv_dtype=c.kv_dtype,
                                        page_size=c.page_size, **strides)
        oracle.paged_prefill(c.q[o0:o0 + n], kp, vp, pt, offs, pos, kv_dtype=c.kv_dtype,
                             n_kv_heads=c.n_kv_heads, page_size=c.page_size, scale=c.scale,
                             **strides)
        f = 4.0 * c.n_heads * c.head_dim * (n * ps + n * (n + 1) // 2)
        return time.perf_counter() - t0, f

    n0 = min(4, ntok)
    t, _ = run(n0)
    n = int(min(ntok, max(n0, n0 * target_s / max(t, 1e-6))))
    t, f = run(n)
    return _cpu_line(f / t / 1e12, "TFLOP/s",
                     f"append and attention of the first {n} of {ntok} new tokens of one sequence "
                     f"after {ps} cached ({f / 1e9:.1f} GFLOP, {t:.1f} s)")


def run_reference(args, case) -> None:
    """--impl reference: the oracle, as it stands, on bounded samples of the workload."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    n = 512
    for _ in range(args.warmup):
        oracle_prefill_sample(case, 32)
    times, flops = [], []
    for s in range(args.steps):
        t, f = oracle_prefill_sample(case, n, seed=100 + s)
        times.append(t)
        flops.append(f)
    value = sum(flops) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "sample_per_step": f"{n} (row, head) outputs"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{n} random (query row, head) outputs per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
# Workloads for profiler captures: the bench's own prefill and verify workloads, and a
# 16-sequence decode (two 1 GiB page pools) that stays a few GB on the device.
CAPTURE_CASES = {
    "prefill_d256": lambda w: w.prefill_d256(seed=0),
    "prefill_d512": lambda w: w.prefill_d512_prefix(seed=0),
    "decode_16seq": lambda w: w.paged_decode(num_seqs=16, num_pages=16384, seed=0),
    "verify": lambda w: w.verify_full(seed=0),
    "verify_fused": lambda w: w.verify_full(seed=0),
    "paged_chunk": lambda w: w.paged_chunk_full(seed=0),
}


def run_capture(name: str, reps: int) -> None:
    import torch
    import workloads
    import attention_gqa_flash_gb300 as g
    torch.cuda.set_device(0)
    g.library()
    c = CAPTURE_CASES[name](workloads)
    if name.startswith("prefill"):
        step = setup_prefill(torch, g, c)[0]
    elif name.startswith("decode"):
        step = setup_decode(torch, g, c)[0]
    elif name == "paged_chunk":
        step = setup_chunk(torch, g, c)[0]
    elif name == "verify_fused":
        fused = setup_verify(torch, g, c)[2]["fused"]

        def step():
            for f in fused.values():
                f()
    else:
        step = setup_verify(torch, g, c)[0]
    for _ in range(max(1, reps)):
        step()
    torch.cuda.synchronize()
    print(f"capture {name}: {max(1, reps)} calls done", flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--paths", choices=("all", "main"), default="all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--capture", choices=tuple(CAPTURE_CASES),
                    help="run one hot-path call --steps times on a capture-sized workload and "
                         "exit (for ncu); prints no JSON line")
    args = ap.parse_args()
    if args.capture:
        run_capture(args.capture, args.steps)
        return
    if args.warmup < 3:
        args.warmup = 3

    import workloads
    head = workloads.prefill_d256(seed=0)
    if args.impl == "reference":
        run_reference(args, head)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import attention_gqa_flash_gb300 as g
    g.library()
    pk, peak_src = peaks()
    tensor_peak = float(pk.get("bf16_tflops", FALLBACK["bf16_tflops"]))
    tensor_peak_sustained = float(pk.get("bf16_tflops_sustained", tensor_peak))
    hbm_peak = float(pk.get("hbm_gbs", FALLBACK["hbm_gbs"]))
    tm = Timer(torch, dist)

    # ---- headline: prefill d256
    step, e2e_step, info = setup_prefill(torch, g, head)
    with Clocks(local) as clk:
        ms = tm.steps(step, args.steps, args.warmup)
    ms_step = tm.max_over_ranks(sum(ms) / len(ms))
    value = world * info["flops"] / (ms_step * 1e-3) / 1e12
    kern = tm.kernel_ms(g, step, max(10, args.steps))
    achieved = info["flops"] / (kern * 1e-3) / 1e12
    # end to end through the public call, eagerly (host copies, marshalling and launches
    # included): one step at a time, and double-buffered (the reported figure)
    e2e_serial = tm.max_over_ranks(sum(tm.steps(e2e_step, args.steps, args.warmup, graph=False)) / args.steps)
    pipe = e2e_step.pipe()
    tm.barrier()
    e2e_ms = tm.max_over_ranks(pipe.run(args.steps, args.warmup))
    del pipe
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded NumPy: Q ~ N(0, 1/16) f32, K/V ~ N(0,1) f16, causal mask)",
        "config": {"workload": head.name, "rows": head.rows, "kv_len": head.kv_len,
                   "n_heads": head.n_heads, "n_kv_heads": head.n_kv_heads,
                   "head_dim": head.head_dim, "scale": head.scale,
                   "flops_per_step": info["flops"],
                   "l2": "flushed before every timed step (512 MiB device write)",
                   "launch": "each step replayed as a CUDA graph of its library calls" if tm.graphs_used
                             else "eager library calls",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "attn_kernel<256,f16>", "achieved": achieved,
                     "peak": tensor_peak, "unit": "TFLOP/s", "frac": achieved / tensor_peak,
                     "kernel_ms": kern,
                     "peak_source": f"{peak_src} bf16_tflops (burst); f16 dense rate equals bf16",
                     "traffic": traffic_for("attn_kernel<256,f16>", head.name)},
        "e2e": {"value": world * info["flops"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": info["h2d"],
                "d2h_bytes_per_step": info["d2h"],
                "pipeline": "double-buffered: each step's host-to-device copy overlaps the "
                            "previous step's attention and device-to-host copy",
                "serial_ms_per_step": e2e_serial},
        # every launch of this library's kernels inside a timed region: the device-timed
        # steps, the kernel timing replays and the end-to-end steps (serial and pipelined)
        "gpu_launches": info["launches"] * (args.steps + max(10, args.steps) + 2 * args.steps),
        "clocks": clk.summary(),
    }
    del step, e2e_step
    torch.cuda.empty_cache()

    # the oracle beside each path, on rank 0 of a single-GPU run (after that path's GPU timing)
    cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if args.paths == "all":
        paths = {}
        # prefill d512 with a 7168-token prefix
        c512 = workloads.prefill_d512_prefix(seed=0)
        s512, _e512, i512 = setup_prefill(torch, g, c512)
        ms = tm.steps(s512, max(5, args.steps // 2), args.warmup)
        t = tm.max_over_ranks(sum(ms) / len(ms))
        k = tm.kernel_ms(g, s512, 5)
        e512 = tm.max_over_ranks(sum(tm.steps(_e512, max(5, args.steps // 2), args.warmup, graph=False))
                                 / max(5, args.steps // 2))
        paths["prefill_d512_prefix"] = {
            "workload": c512.name, "value": world * i512["flops"] / (t * 1e-3) / 1e12,
            "unit": "TFLOP/s", "ms_per_step": t,
            "e2e": {"value": world * i512["flops"] / (e512 * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": e512, "h2d_bytes_per_step": i512["h2d"],
                    "d2h_bytes_per_step": i512["d2h"], "pipeline": "serial: one step at a time"},
            "roofline": {"bound": "tensor", "kernel": "attn_kernel<512,f16>",
                         "achieved": i512["flops"] / (k * 1e-3) / 1e12, "peak": tensor_peak,
                         "unit": "TFLOP/s", "frac": i512["flops"] / (k * 1e-3) / 1e12 / tensor_peak,
                         "kernel_ms": k, "traffic": traffic_for("attn_kernel<512,f16>", c512.name),
                         "note": "two output halves recompute Q.K^T: executed FLOPs are 1.5x"}}
        if cpu:
            paths["prefill_d512_prefix"]["cpu_baseline"] = cpu_prefill(c512)
        del s512, _e512
        torch.cuda.empty_cache()
        # paged decode
        dc = workloads.paged_decode(seed=0)
        sd, idc = setup_decode(torch, g, dc)
        ms = tm.steps(sd, max(5, args.steps // 2), args.warmup)
        t = tm.max_over_ranks(sum(ms) / len(ms))
        k = tm.kernel_ms(g, sd, 5)
        e2e_fn, hi, ho = idc["e2e"]
        ed = tm.max_over_ranks(sum(tm.steps(e2e_fn, max(5, args.steps // 2), args.warmup, graph=False))
                               / max(5, args.steps // 2))
        paths["paged_decode"] = {
            "workload": dc.name, "value": world * idc["bytes"] / (t * 1e-3) / 1e9, "unit": "GB/s",
            "kv_bytes_per_step": idc["kv_bytes"], "ms_per_step": t,
            "e2e": {"value": world * idc["bytes"] / (ed * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ed,
                    "h2d_bytes_per_step": hi, "d2h_bytes_per_step": ho,
                    "pipeline": "serial: one step at a time; the KV pools are the resident cache"},
            "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel<f16,128>",
                         "achieved": idc["kernel_bytes"] / (k * 1e-3) / 1e9, "peak": hbm_peak,
                         "unit": "GB/s", "frac": idc["kernel_bytes"] / (k * 1e-3) / 1e9 / hbm_peak,
                         "kernel_ms": k, "traffic": traffic_for("paged_decode_kernel<f16,128>", dc.name)}}
        if cpu:
            paths["paged_decode"]["cpu_baseline"] = cpu_decode(dc)
        del sd, dc, e2e_fn, idc
        torch.cuda.empty_cache()
        # speculative verify chain
        vc = workloads.verify_full(seed=0)
        sv, ops, iv = setup_verify(torch, g, vc)
        ms = tm.steps(sv, max(5, args.steps // 2), args.warmup)
        t = tm.max_over_ranks(sum(ms) / len(ms))
        total = sum(iv["bytes"].values())
        kernels = {}
        for name, f in ops.items():
            k = tm.kernel_ms(g, f, 5)
            kernels[name] = {"bytes": iv["bytes"][name], "kernel_ms": k,
                             "achieved_gbs": iv["bytes"][name] / (k * 1e-3) / 1e9,
                             "frac": iv["bytes"][name] / (k * 1e-3) / 1e9 / hbm_peak}
        e2e_fn, hi, ho = iv["e2e"]
        ev_ = tm.max_over_ranks(sum(tm.steps(e2e_fn, max(5, args.steps // 2), args.warmup, graph=False))
                                / max(5, args.steps // 2))
        paths["verify_chain"] = {"workload": vc.name, "value": world * total / (t * 1e-3) / 1e9,
                                 "unit": "GB/s", "ms_per_step": t, "bytes_per_step": total,
                                 "peak": hbm_peak, "frac": total / (t * 1e-3) / 1e9 / hbm_peak,
                                 "kernels": kernels,
                                 "e2e": {"value": world * total / (ev_ * 1e-3) / 1e9, "unit": "GB/s",
                                         "ms_per_step": ev_, "h2d_bytes_per_step": hi,
                                         "d2h_bytes_per_step": ho,
                                         "pipeline": "serial: one step at a time; the rings are the "
                                                     "resident cache"}}
        # the same verify step with the fused ring-direct attention (no pack, no mask)
        fops, fby = iv["fused"], iv["fused_bytes"]

        def fstep():
            for f in fops.values():
                f()
        ms = tm.steps(fstep, max(5, args.steps // 2), args.warmup)
        t = tm.max_over_ranks(sum(ms) / len(ms))
        ftotal = sum(fby.values())
        fkernels = {}
        for name, f in fops.items():
            k = tm.kernel_ms(g, f, 5)
            fkernels[name] = {"bytes": fby[name], "kernel_ms": k,
                              "achieved_gbs": fby[name] / (k * 1e-3) / 1e9,
                              "frac": fby[name] / (k * 1e-3) / 1e9 / hbm_peak}
        fkernels["attn"]["traffic"] = traffic_for("attn_kernel<256,bf16,ring>", vc.name)
        e2e_fn, hi, ho = iv["fused_e2e"]
        ef = tm.max_over_ranks(sum(tm.steps(e2e_fn, max(5, args.steps // 2), args.warmup, graph=False))
                               / max(5, args.steps // 2))
        paths["verify_fused"] = {"workload": vc.name, "value": world * ftotal / (t * 1e-3) / 1e9,
                                 "unit": "GB/s", "ms_per_step": t, "bytes_per_step": ftotal,
                                 "peak": hbm_peak, "frac": ftotal / (t * 1e-3) / 1e9 / hbm_peak,
                                 "kernels": fkernels,
                                 "e2e": {"value": world * ftotal / (ef * 1e-3) / 1e9, "unit": "GB/s",
                                         "ms_per_step": ef, "h2d_bytes_per_step": hi,
                                         "d2h_bytes_per_step": ho,
                                         "pipeline": "serial: one step at a time; the rings are the "
                                                     "resident cache"}}
        if cpu:
            paths["verify_chain"]["cpu_baseline"], paths["verify_fused"]["cpu_baseline"] = \
                cpu_verify(vc, total, ftotal)
        verify_launches, fused_launches = iv["launches"], iv["fused_launches"]
        del sv, ops, fops, fstep, vc, iv, e2e_fn
        torch.cuda.empty_cache()
        # chunked prefill over pages: page append + attention
        cc = workloads.paged_chunk_full(seed=0)
        sc, cops, ic = setup_chunk(torch, g, cc)
        ms = tm.steps(sc, max(5, args.steps // 2), args.warmup)
        t = tm.max_over_ranks(sum(ms) / len(ms))
        ka = tm.kernel_ms(g, cops["append"], 5)
        kt = tm.kernel_ms(g, cops["attn"], 5)
        e2e_fn, hi, ho = ic["e2e"]
        ec = tm.max_over_ranks(sum(tm.steps(e2e_fn, max(5, args.steps // 2), args.warmup, graph=False))
                               / max(5, args.steps // 2))
        paths["paged_chunk_prefill"] = {
            "workload": cc.name, "value": world * ic["flops"] / (t * 1e-3) / 1e12,
            "unit": "TFLOP/s", "ms_per_step": t, "flops_per_step": ic["flops"],
            "e2e": {"value": world * ic["flops"] / (ec * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ec,
                    "h2d_bytes_per_step": hi, "d2h_bytes_per_step": ho,
                    "pipeline": "serial: one step at a time (append and attention); the page pools "
                                "are the resident cache"},
            "roofline": {"bound": "tensor", "kernel": "attn_kernel<256,f16,paged>",
                         "achieved": ic["flops"] / (kt * 1e-3) / 1e12, "peak": tensor_peak,
                         "unit": "TFLOP/s", "frac": ic["flops"] / (kt * 1e-3) / 1e12 / tensor_peak,
                         "kernel_ms": kt, "traffic": traffic_for("attn_kernel<256,f16,paged>", cc.name)},
            "append": {"kernel": "page_append_kernel<f16>", "bytes": ic["append_bytes"],
                       "traffic": traffic_for("page_append_kernel<f16>", cc.name),
                       "kernel_ms": ka, "achieved_gbs": ic["append_bytes"] / (ka * 1e-3) / 1e9,
                       "frac": ic["append_bytes"] / (ka * 1e-3) / 1e9 / hbm_peak}}
        if cpu:
            paths["paged_chunk_prefill"]["cpu_baseline"] = cpu_chunk(cc)
        chunk_launches = ic["launches"]
        del sc, cops, cc, ic, e2e_fn
        torch.cuda.empty_cache()
        line["paths"] = paths
        # per path: device-timed steps and end-to-end steps (n each), and the kernel timing
        # replays (5 per timed kernel)
        n = max(5, args.steps // 2)
        line["gpu_launches"] += (2 * (2 * n + 5) + 2 * (2 * n + 5) + verify_launches * 2 * n + 5 * 4
                                 + fused_launches * 2 * n + 5 * 2 + chunk_launches * 2 * n + 5 * 2)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(head)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
