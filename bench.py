#!/usr/bin/env python3
"""Benchmark of the paged GQA decode + block scoring + eviction gather path.

One step = append one token per sequence -> paged split-K GQA decode with
per-block mass -> EMA / priority / tier scoring -> selection of P < 0.3
blocks -> gather of their pages to pinned host memory.  Metric: KV bytes
streamed per second (GB/s), with decode tokens/s alongside.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed

Multi-GPU: replicas only (one independent pool per rank, no collective on
the data path); launched by torchrun, value = all ranks' bytes / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV GB/s streamed (% of GB300 HBM peak) + decode tok/s, paged GQA decode+scoring"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_dram_traffic.txt")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvs", "reference"], default="kvs")
    ap.add_argument("--workload", default="l70b_128k")
    ap.add_argument("--alpha", type=float, default=None)
    ap.add_argument("--gather", choices=["auto", "mirror", "mirror-sync", "list", "demote", "prefetch", "ids",
                                         "ids-sync", "none"],
                    default="auto",
                    help="auto: demote for workloads with periodic demotion, else mirror (ids in 2-bit "
                         "contexts); mirror / ids: the asynchronous select (no host wait per step), "
                         "mirror-sync / ids-sync: the synchronising one; prefetch: demoted blocks "
                         "come back in fetch order, a budget per step, while the sequences without "
                         "holes decode")
    ap.add_argument("--prefetch-budget", type=int, default=512,
                    help="blocks re-admitted per step in prefetch mode")
    ap.add_argument("--victims", choices=["lowfrac", "lrfu"], default="lowfrac",
                    help="demotion victims: smallest P, or smallest LRFU key (lazily decayed "
                         "EMA of touches)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8", "kivi2"], default="bf16",
                    help="page element type: bf16, FP8 E4M3 codes (per-tensor scale 1.0), or 2-bit "
                         "groups behind a 128-token bf16 residual window")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-literal", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="decode and score in two calls (kvs_decode_step + kvs_score_update) instead of "
                         "kvs_decode_score_step")
    ap.add_argument("--no-batched", action="store_true",
                    help="128K workload only: skip the batched workload's line under \"batched\"")
    ap.add_argument("--cpu-layers", type=int, default=8,
                    help="layers of the workload in the CPU-baseline sample")
    ap.add_argument("--decode-event-every", type=int, default=4,
                    help="record the decode kernel's CUDA event pair on every Nth timed step (1: all). "
                         "An event between the decode-set upload and the decode launch makes that "
                         "step's decode a plain launch, so the other steps carry none")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling cut: the workload's first N layers only (same sequences; a "
                         "decode launch's reads scale by L / N).  Not a bench figure of the named "
                         "workload (its line carries no traffic figure)")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def session_copy_rate(torch, dev, gib=4, reps=20):
    """The box's streaming copy rate in this session ([VA] method for its copy
    figure: large buffers, median of repeated runs): a device-to-device copy
    of `gib` GiB, read + write bytes, the median of `reps` runs timed with
    CUDA events."""
    n = (gib << 30) // 2
    a = torch.empty(n, dtype=torch.bfloat16, device=dev).normal_()
    b = torch.empty_like(a)
    b.copy_(a)
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    del a, b
    torch.cuda.empty_cache()
    return 2 * n * 2 / (statistics.median(ts) / 1e3) / 1e9


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# kernel sources whose code decides the DRAM traffic of each page format's decode
TRAFFIC_SOURCES = {
    "bf16": ("kvs_decode.cu", "kvs_ptx.h", "kvs_internal.h"),
    "fp8": ("kvs_decode.cu", "kvs_ptx.h", "kvs_internal.h"),
    "kivi2": ("kvs_decode.cu", "kvs_kivi.cu", "kvs_ptx.h", "kvs_internal.h"),
}


def decode_source_hash(kv_dtype):
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[kv_dtype]:
        with open(os.path.join(ROOT, "paged_kv_cache_flash_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(workload, kv_dtype):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source for this workload
    and page format."""
    try:
        txt = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    src = re.search(rf"source_hash\[{re.escape(kv_dtype)}\]:\s*(\S+)", txt)
    if not src or src.group(1) != decode_source_hash(kv_dtype):
        return None
    key = workload + ("" if kv_dtype == "bf16" else "_" + kv_dtype)
    m = re.search(rf"traffic_bytes_per_launch\[{re.escape(key)}\]:\s*([0-9.eE+]+)", txt)
    return float(m.group(1)) if m else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a region."""
    Q = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import torch
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid).lower()
        except Exception:
            pass
        self.proc = None
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "20"]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        uuids = {r[0].lower() for r in rows}
        if len(uuids) > 1 and self.uuid:
            rows = [r for r in rows if self.uuid in r[0].lower()] or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows
                                    if re.match(r"^[0-9.]+$", r[3])), default=None)}


def reduce_over_ranks(ms: float, nbytes: float, device=None):
    """Replicas: the job's time is the slowest rank's, its bytes the sum of
    every rank's.  Returns (max ms, total bytes); identity without a process
    group.  `device`: where the reduction tensors live (cuda for NCCL, cpu
    for gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms), float(nbytes)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


# --------------------------------------------------------------- kvs arm


class Pipeline:
    """The hot path, driven through the public C ABI for a set of sequences."""

    def __init__(self, wl, alpha, steps_total, device, gather, kv_dtype="bf16", prefetch_budget=512,
                 victims="lowfrac", fused=True):
        import torch
        import paged_kv_cache_flash_gb300 as K
        import workloads as W
        self.torch, self.K, self.W = torch, K, W
        self.wl, self.dev, self.gather = wl, device, gather
        self.fused = fused
        B = wl.block_tokens
        self.ids = [5000 - 17 * s for s in range(wl.nseq)]
        self.ntok = list(wl.prefill_lens)
        mb = max((n + steps_total + B - 1) // B for n in wl.prefill_lens) + 1
        need = sum((n + steps_total + B - 1) // B for n in wl.prefill_lens)
        need -= (wl.shared_prefix_tokens // B) * (wl.nseq - 1)
        self.pool_pages = max(wl.pool_pages, need + 8)
        self.kivi = kv_dtype == "kivi2"
        groups = 0
        if self.kivi:
            # bf16 pages hold the residual windows (at most 160 + 15 tokens each)
            # and one prefill chunk in flight; group pages hold the rest
            self.pool_pages = wl.nseq * 12 + self.PREFILL_CHUNK // B + 16
            groups = sum((n + steps_total) // K.KVS_KIVI_GROUP_TOKENS for n in wl.prefill_lens) + wl.nseq
        dt = {"bf16": K.KVS_KV_BF16, "fp8": K.KVS_KV_FP8_E4M3, "kivi2": K.KVS_KV_KIVI2}[kv_dtype]
        cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, self.pool_pages, wl.nseq, mb, alpha=alpha,
                            recency_window=wl.recency_window, weights=wl.weights, cuts=wl.cuts,
                            pool_seed=wl.seed, staging_pages=32, kv_dtype=dt, kivi_groups=groups)
        self.ctx = K.Context(cfg, device)
        self.token_bytes = wl.token_bytes // (2 if kv_dtype == "fp8" else 1)
        # 2-bit groups: 3 KiB per (layer, KV head) and 32 tokens
        self.group_token_bytes = wl.L * wl.Hkv * 3072 // 32
        self.side = torch.cuda.Stream(device)
        self.out = torch.empty((wl.nseq, wl.L, wl.Hq, wl.d), dtype=torch.float32, device=device)
        self.host = None
        self.demote_every = wl.demote_every if gather in ("demote", "prefetch") else 0
        self.steps_done = 0
        self.demoted_pages = 0
        self.prefetched_pages = 0
        self.holes = {}                     # prefetch: seq_id -> blocks still demoted
        self.budget = prefetch_budget
        self.last_round = 0                 # pages demoted by the last step (0: none)
        self.victim_mode = K.KVS_SELECT_LRFU if victims == "lrfu" else K.KVS_SELECT_LOWFRAC
        self.pf_stream = torch.cuda.Stream(device) if gather == "prefetch" else None
        self.pf_done = None
        self.async_pending = False          # an asynchronous select's counts are due
        self.async_staged = 0
        self.all_idx = list(range(wl.nseq))
        self.active = self.all_idx          # sequences decoded by the last step
        self._idx = {}
        if gather in ("mirror", "mirror-sync", "list"):
            self.host = torch.empty(self.pool_pages * self.ctx.page_bytes, dtype=torch.uint8,
                                    pin_memory=True)
        elif gather in ("demote", "prefetch"):
            k_max = int(math.floor(wl.demote_frac * (need + wl.nseq))) + 1
            self.host = torch.empty(k_max * self.ctx.page_bytes, dtype=torch.uint8, pin_memory=True)
            self.ids_dev = torch.zeros(2 * (need + wl.nseq), dtype=torch.int64, device=device)
        if self.host is not None:
            # set-up: the first copy-engine transfer into fresh pinned memory maps
            # it (about 2/3 of the warm rate); do that once here rather than inside
            # the first timed gather or demotion
            z = torch.zeros(1 << 30, dtype=torch.uint8, device=device)
            for a in range(0, self.host.numel(), z.numel()):
                n = min(z.numel(), self.host.numel() - a)
                self.host[a:a + n].copy_(z[:n])
            torch.cuda.synchronize()
            del z

    PREFILL_CHUNK = 4096

    def prefill(self, chunk=PREFILL_CHUNK):
        wl, W = self.wl, self.W
        # 2-bit group contexts share no pages: each sequence holds its own prefix
        pre = 0 if self.kivi else wl.shared_prefix_tokens // wl.block_tokens
        for s, sid in enumerate(self.ids):
            if s > 0 and pre:
                self.ctx.seq_add(sid, self.ids[0], pre)
                start = wl.shared_prefix_tokens
            else:
                self.ctx.seq_add(sid)
                start = 0
            for a in range(start, wl.prefill_lens[s], chunk):
                b = min(wl.prefill_lens[s], a + chunk)
                Kt, Vt = W.kv_tokens(wl, s, a, b, self.dev)
                self.ctx.append_tokens(sid, Kt, Vt)
                del Kt, Vt
        self.torch.cuda.synchronize()

    def inputs(self, step0, nsteps):
        """Per-step new-token K/V ([nseq][L][Hkv][d] each) and queries, generated
        on the device."""
        wl, W, torch = self.wl, self.W, self.torch
        kv, qs = [], []
        for i in range(nsteps):
            t = step0 + i
            ks, vs = [], []
            for s in range(wl.nseq):
                n = wl.prefill_lens[s] + t - 1
                k, v = W.kv_tokens(wl, s, n, n + 1, self.dev)
                ks.append(k)
                vs.append(v)
            kv.append((torch.cat(ks).contiguous(), torch.cat(vs).contiguous()))
            qs.append(torch.stack([W.queries(wl, s, t, self.dev) for s in range(wl.nseq)]).contiguous())
        return kv, qs

    def kv_bytes_this_step(self):
        # bytes of the tokens attended (after append) by the sequences decoded this step
        if self.kivi:
            tot = 0
            for i in self.active:
                n = self.ntok[i]
                q = 32 * (max(0, n - 128) // 32)
                tot += q * self.group_token_bytes + (n - q) * self.token_bytes
            return tot
        return sum(self.ntok[i] for i in self.active) * self.token_bytes

    def _rows(self, x, active):
        if len(active) == len(self.ids):
            return x
        key = tuple(active)
        if key not in self._idx:
            self._idx[key] = self.torch.tensor(active, dtype=self.torch.int64, device=self.dev)
        return x.index_select(0, self._idx[key])

    def step(self, kv_row, q, ev=None, mode_flags=None, after_decode=None, phases=True):
        """One decode step.  ev: 5 timing events (step start, after append,
        after decode, after score, step end); with phases=False only a demote
        round records two of them (after score, step end), so that nothing
        sits between the kernels of the other steps or between steps (an
        event in the stream stops the next kernel's programmatic early
        launch)."""
        K, ctx, torch = self.K, self.ctx, self.torch
        main = torch.cuda.current_stream()
        sh, side = main.cuda_stream, self.side.cuda_stream    # raw handles: no lookups per call
        if ev and phases:
            ev[0].record(main)
        paused = set()
        if self.gather == "prefetch":
            # blocks re-admitted by the last step are in place before anything reads them
            if self.pf_done is not None:
                main.wait_event(self.pf_done)
            paused = set(self.holes)
            if self.holes:
                # plan first (its kernel cannot share the SMs with the decode),
                # then the copies run on their own stream beside this step's decode
                plan = ctx.prefetch(self.budget, self.host, stream=self.pf_stream)
                done = torch.cuda.Event()
                done.record(self.pf_stream)
                self.pf_done = done
                for sid, _, _, _ in plan:
                    self.holes[sid] -= 1
                self.holes = {k: v for k, v in self.holes.items() if v > 0}
                self.prefetched_pages += len(plan)
        if paused:
            active = [i for i, sid in enumerate(self.ids) if sid not in paused]
            ids = [self.ids[i] for i in active]
            out = self.out[:len(active)]
        else:
            active, ids, out = self.all_idx, self.ids, self.out
        self.active = active
        ctx.append_step(ids, self._rows(kv_row[0], active), self._rows(kv_row[1], active), stream=sh)
        for i in active:
            self.ntok[i] += 1
        if ev and phases:
            ev[1].record(main)
        if self.fused:      # scoring in the decode epilogue
            ctx.decode_score_step(ids, self._rows(q, active), out, stream=sh)
        else:
            ctx.decode_step(ids, self._rows(q, active), out, stream=sh)
        if ev and phases:
            ev[2].record(main)
        if after_decode is not None:
            after_decode()          # host work that overlaps the rest of the step
        if not self.fused:
            ctx.score_update(stream=sh)
        r = None
        self.steps_done += 1
        demoting = self.demote_every and self.steps_done % self.demote_every == 0 and not self.holes
        if ev and (phases or demoting):
            ev[3].record(main)
        if self.gather in ("ids", "ids-sync"):      # the THRESH list only, no page copies
            flags = K.KVS_GATHER_ASYNC if self.gather == "ids" else 0
            r = self._select(K.KVS_SELECT_THRESH, None, flags, sh, sh)
        elif self.gather in ("mirror", "mirror-sync", "list"):
            flags = {"mirror": K.KVS_GATHER_MIRROR | K.KVS_GATHER_ASYNC,
                     "mirror-sync": K.KVS_GATHER_MIRROR, "list": 0}[self.gather]
            if mode_flags is not None:
                flags = mode_flags
            r = self._select(K.KVS_SELECT_THRESH, self.host, flags, sh, side)
            if not flags & K.KVS_GATHER_ASYNC:
                main.wait_stream(self.side)
        elif self.demote_every and self.steps_done % self.demote_every == 0 and not self.holes:
            # the lowest-P fraction goes to pinned host and comes back with its record
            rc, r = ctx.select_and_gather(self.victim_mode, self.host, frac=self.wl.demote_frac,
                                          flags=K.KVS_GATHER_DEMOTE, ids=self.ids_dev,
                                          side_stream=self.side)
            keys = [tuple(x) for x in self.ids_dev.view(-1, 2)[: r.n_demoted].cpu().tolist()]
            self.demoted_pages += r.n_demoted
            self.last_round = r.n_demoted
            if self.gather == "demote":
                ctx.readmit(keys, self.host)        # overlaps the demotion's copies
                main.wait_stream(self.side)
            else:
                for sid, _ in keys:
                    self.holes[sid] = self.holes.get(sid, 0) + 1
        if ev and (phases or demoting):
            ev[4].record(main)
        return r


    def _select(self, mode, host, flags, stream, side):
        """THRESH select; an asynchronous call returns None and its counts are
        collected at the next select (or by flush_counts), so the host never
        waits for the step it has just enqueued."""
        K, ctx = self.K, self.ctx
        if self.async_pending:
            self.async_staged += ctx.gather_counts().n_staged
            self.async_pending = False
        rc, r = ctx.select_and_gather(mode, host, flags=flags, stream=stream, side_stream=side)
        if flags & K.KVS_GATHER_ASYNC:
            self.async_pending = True
            return None
        return r

    def flush_counts(self):
        """Pages staged by asynchronous selects whose counts are not yet in."""
        if self.async_pending:
            self.async_staged += self.ctx.gather_counts().n_staged
            self.async_pending = False
        n, self.async_staged = self.async_staged, 0
        return n


def cpu_sample(wl, n_tokens, layers, device):
    """K, V of the first `layers` layers of sequence 0 (all tokens), and the
    step-1 query of those layers, as host tensors, from the generator."""
    import torch
    import workloads as W
    Ks, Vs = [], []
    for a in range(0, n_tokens, 4096):
        b = min(n_tokens, a + 4096)
        Kt, Vt = W.kv_tokens(wl, 0, a, b, device)
        Ks.append(Kt[:, :layers].cpu())
        Vs.append(Vt[:, :layers].cpu())
        del Kt, Vt
    q = W.queries(wl, 0, 1, device)[:layers].cpu()
    return q, torch.cat(Ks).contiguous(), torch.cat(Vs).contiguous()


def time_oracle(wl, q, K, V, layers, threads):
    import oracle as O
    t0 = time.perf_counter()
    O.decode(q, K, V, L=layers, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, threads=threads,
             want_out=True, want_head_mass=True)
    return time.perf_counter() - t0


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_leg(wl, dev, layers, alpha, kv_bytes_step, pages_step):
    """The oracle, as it stands, timed on this host's cores on bounded samples
    of one step of the workload, and the whole step estimated from them:
    attention + block mass (fp64, the C oracle) of sequence 0 on `layers` of
    its layers with every core and on one layer with one thread, scaled to
    all layers and sequences by tokens; then the scoring, THRESH selection
    and gather plan of every record of the workload (numpy, one thread), and
    the page assembly of 8 pages (scaled to the pages the path sends to the
    host per step)."""
    import numpy as np
    import oracle as O
    import workloads as W
    n = wl.prefill_lens[0] + 1
    q, Kc, Vc = cpu_sample(wl, n, layers, dev)
    allc = os.cpu_count() or 1
    t_all = time_oracle(wl, q, Kc, Vc, layers, allc) / layers
    K1, V1 = Kc[:, :1].contiguous(), Vc[:, :1].contiguous()
    t_one = time_oracle(wl, q[:1].contiguous(), K1, V1, 1, 1)
    tok_total = sum(x + 1 for x in wl.prefill_lens)
    attn_all = t_all * wl.L * tok_total / n
    attn_one = t_one * wl.L * tok_total / n
    B = wl.block_tokens
    recs = {5000 - 17 * s: O.new_records(5000 - 17 * s, 0, (x + B) // B, 0)
            for s, x in enumerate(wl.prefill_lens)}
    masses = {sid: W.synthetic_masses(sid, len(r)).astype(np.float64) for sid, r in recs.items()}
    t0 = time.perf_counter()
    recs = {sid: O.score_update(r, masses[sid], 1, alpha, wl.recency_window, wl.weights, wl.cuts)
            for sid, r in recs.items()}
    t_score = time.perf_counter() - t0
    t0 = time.perf_counter()
    ids = O.select_thresh(recs)
    page_of = {k: k for k in ids}
    O.gather_plan(ids, page_of, {k: {k} for k in ids})
    t_select = time.perf_counter() - t0
    npg = min(8, n // B)
    t0 = time.perf_counter()
    for b in range(npg):
        O.assemble_page(Kc[b * B:(b + 1) * B], Vc[b * B:(b + 1) * B], B)
    t_page = (time.perf_counter() - t0) / max(npg, 1) * wl.L / layers
    rest = t_score + t_select + t_page * pages_step
    step_all, step_one = attn_all + rest, attn_one + rest
    return {"value": round(kv_bytes_step / step_all / 1e9, 4), "unit": UNIT, "cores": allc, "kind": "oracle",
            "cpu_model": cpu_model(),
            "single_thread": {"value": round(kv_bytes_step / step_one / 1e9, 4), "unit": UNIT, "cores": 1},
            "step_estimate_s": {"all_cores": round(step_all, 3), "one_thread": round(step_one, 3)},
            "parts_s": {"attention_per_layer_seq0_all_cores": round(t_all, 4),
                        "attention_per_layer_seq0_one_thread": round(t_one, 4),
                        "score_all_records": round(t_score, 4), "select_and_plan": round(t_select, 4),
                        "page_assembly_per_page": round(t_page, 5), "pages_per_step": round(pages_step, 2)},
            "sample": f"sequence 0 ({n} tokens): fp64 attention + block mass of layers 0..{layers - 1} "
                      f"of {wl.L} on {allc} threads and of layer 0 on 1 thread, scaled by layers and "
                      f"tokens to the step ({tok_total} tokens); scoring, THRESH selection and gather "
                      f"plan of all {sum(len(r) for r in recs.values())} records; page assembly of "
                      f"{npg} pages x the {pages_step:.1f} pages the path sends to host per step"}


def measure(args, wname, dev, ws, rank, local, sub=False):
    """Times K steps of one workload after W warm-up steps and returns the
    JSON fields of its line (rank 0; None elsewhere).  sub: a second workload
    of the same run -- no literal-gather, copy-rate or CPU-baseline legs."""
    import torch
    import workloads as W
    wl = W.workload(wname)
    if args.layers:
        wl = wl.with_(L=args.layers)
    alpha = args.alpha if args.alpha is not None else wl.alphas[-1]
    gather = args.gather
    if gather == "auto":
        gather = "ids" if args.kv_dtype == "kivi2" else ("demote" if wl.demote_every else "mirror")
    K_, W_ = args.steps, args.warmup
    e2e_steps = 0 if args.no_e2e else K_
    lit_steps = 0 if (sub or args.no_literal or gather not in ("mirror", "mirror-sync", "list")) else 2
    bd_steps = min(8, K_)
    total = W_ + K_ + bd_steps + e2e_steps + lit_steps
    pipe = Pipeline(wl, alpha, total, dev, gather, args.kv_dtype, args.prefetch_budget, args.victims,
                    fused=not args.unfused)
    pipe.prefill()
    kv, qs = pipe.inputs(1, W_ + K_)

    for i in range(W_):
        pipe.step(kv[i], qs[i])
    pipe.flush_counts()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K_)]
    dec = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K_)]
    for e in dec:
        for x in e:
            x.record()
    torch.cuda.synchronize()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    kv_bytes = 0
    decoded = 0                     # sequence-steps decoded (all, unless prefetch pauses some)
    uniq_bytes = 0
    staged = 0
    shared_extra = 0 if pipe.kivi else wl.shared_prefix_tokens * (wl.nseq - 1) * pipe.token_bytes
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = pipe.ctx.kernel_launches()
    prefetched0 = pipe.prefetched_pages
    demoted0 = pipe.demoted_pages
    wall0 = time.perf_counter()
    t_start.record()
    rounds = []                     # (timed step, pages) of demote + readmit round trips
    dec_every = max(1, args.decode_event_every)
    dec_steps = [i for i in range(K_) if i % dec_every == 0]
    for i in range(K_):
        if i % dec_every == 0:
            pipe.ctx.set_decode_events(dec[i][0], dec[i][1])
        else:
            pipe.ctx.set_decode_events(None, None)
        pipe.last_round = 0
        r = pipe.step(kv[W_ + i], qs[W_ + i], ev[i], phases=False)
        if pipe.last_round and gather == "demote":
            rounds.append((i, pipe.last_round))
        kv_bytes += pipe.kv_bytes_this_step()
        decoded += len(pipe.active)
        uniq_bytes += pipe.kv_bytes_this_step() - shared_extra
        staged += r.n_staged if r is not None else 0
    demoted = pipe.demoted_pages - demoted0
    t_stop.record()
    torch.cuda.synchronize()
    ntok_timed = list(pipe.ntok)
    staged += pipe.flush_counts()
    wall = time.perf_counter() - wall0
    launches = pipe.ctx.kernel_launches() - launches0
    prefetched = pipe.prefetched_pages - prefetched0
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    pipe.ctx.set_decode_events(None, None)
    pipe.ctx.check_device()
    ms = t_start.elapsed_time(t_stop)

    ms_max, bytes_all = reduce_over_ranks(ms, kv_bytes, dev)
    value = bytes_all / (ms_max / 1e3) / 1e9
    tok_s = decoded * ws / (ms_max / 1e3)

    dec_ms = [dec[i][0].elapsed_time(dec[i][1]) for i in dec_steps]
    round_info = None
    if rounds:
        # selection + demotion (D2H) + re-admission (H2D) region of those steps
        r_ms = [ev[i][3].elapsed_time(ev[i][4]) for i, _ in rounds]
        r_bytes = [2 * n * pipe.ctx.page_bytes for _, n in rounds]
        round_info = {"rounds": len(rounds), "pages_per_round": int(statistics.median(n for _, n in rounds)),
                      "ms_per_round": round(statistics.median(r_ms), 3),
                      "link_GBps": round(sum(r_bytes) / (sum(r_ms) / 1e3) / 1e9, 2),
                      "note": "2 x page bytes per demoted page (to host and back) over the region"}
    # ---- per-phase breakdown: a few more steps with an event between calls
    # (kept out of the timed steps, where the calls' kernels follow each
    # other with nothing in between)
    kvb, qb = pipe.inputs(W_ + K_ + 1, bd_steps)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(bd_steps)]
    for i in range(bd_steps):
        pipe.step(kvb[i], qb[i], evb[i])
    pipe.flush_counts()
    torch.cuda.synchronize()
    del kvb, qb
    part = {name: statistics.median(evb[i][a].elapsed_time(evb[i][b]) for i in range(bd_steps))
            for name, a, b in [("append", 0, 1), ("decode_step", 1, 2), ("score", 2, 3),
                               ("select_gather", 3, 4)]}
    dec_avg = sum(dec_ms) / len(dec_ms)
    B = wl.block_tokens
    nb = [(n + B - 1) // B for n in ntok_timed]
    algo = kv_bytes / K_ + wl.nseq * wl.L * wl.Hq * wl.d * 2 + sum(nb) * 4
    achieved = algo / (dec_avg / 1e3) / 1e9
    peak, peak_src = read_peaks()
    traffic = None if args.layers else read_traffic(wname, args.kv_dtype)

    # ---- end to end through host buffers --------------------------------
    e2e = None
    if e2e_steps:
        pipe.flush_counts()
        kvh, qh = pipe.inputs(W_ + K_ + bd_steps + 1, e2e_steps)
        kvh = [(k.cpu().pin_memory(), v.cpu().pin_memory()) for k, v in kvh]
        qh = [q.cpu().pin_memory() for q in qh]
        # double-buffered: the inputs of step i + 1 go up on one copy stream and
        # the output of step i comes down on another while step i + 1 computes;
        # every copy is inside the timed region
        dkv = [(torch.empty_like(kv[0][0]), torch.empty_like(kv[0][1])) for _ in range(2)]
        dq = [torch.empty_like(qs[0]) for _ in range(2)]
        outs = [pipe.out, torch.empty_like(pipe.out)]
        out_h = torch.empty(pipe.out.shape, dtype=torch.float32, pin_memory=True)
        h2d = kvh[0][0].numel() * 2 + kvh[0][1].numel() * 2 + qh[0].numel() * 2
        d2h = out_h.numel() * 4
        main = torch.cuda.current_stream()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def upload(i):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(done[b])      # step i - 2 has read this buffer
                dkv[b][0].copy_(kvh[i][0], non_blocking=True)
                dkv[b][1].copy_(kvh[i][1], non_blocking=True)
                dq[b].copy_(qh[i], non_blocking=True)
                in_ready[b].record(up)

        def after_decode(i):
            # runs once step i's decode is enqueued, while the device works: its
            # inputs are consumed and its output final on the stream from here
            b = i % 2
            done[b].record(main)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                out_h.copy_(outs[b], non_blocking=True)
                out_free[b].record(down)
            if i + 1 < e2e_steps:
                upload(i + 1)

        torch.cuda.synchronize()
        e_b = 0
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        up.wait_event(s0)
        upload(0)
        for i in range(e2e_steps):
            b = i % 2
            main.wait_event(in_ready[b])
            if i >= 2:
                main.wait_event(out_free[b])
            pipe.out = outs[b]
            pipe.step(dkv[b], dq[b], after_decode=lambda i=i: after_decode(i))
            e_b += pipe.kv_bytes_this_step()
        main.wait_stream(down)
        main.wait_stream(up)
        s1.record()
        torch.cuda.synchronize()
        pipe.out = outs[0]
        e_ms = s0.elapsed_time(s1)
        e_ms_max, e_b_all = reduce_over_ranks(e_ms, e_b, dev)
        e_val = e_b_all / (e_ms_max / 1e3) / 1e9
        e2e = {"value": round(e_val, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e_ms / e2e_steps, 4),
               "copies": "pinned host, double-buffered on two copy streams beside the steps"}

    # ---- literal per-step gather of every P < 0.3 page (list mode) -------
    literal = None
    if lit_steps:
        kvl, ql = pipe.inputs(W_ + K_ + bd_steps + e2e_steps + 1, lit_steps)
        torch.cuda.synchronize()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pages = moved = 0
        lw = time.perf_counter()
        for i in range(lit_steps):
            evl = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            r = pipe.step(kvl[i], ql[i], evl, mode_flags=0)
            torch.cuda.synchronize()
            if i == lit_steps - 1:
                literal_ms = evl[3].elapsed_time(evl[4])
            pages, moved = r.n_pages, r.bytes_to_host
        literal = {"pages_per_step": int(pages), "bytes_to_host_per_step": int(moved),
                   "select_gather_ms": round(literal_ms, 3),
                   "host_link_GBps": round(moved / (literal_ms / 1e3) / 1e9, 2) if literal_ms else None}

    # ---- the box's streaming copy rate in this session (context for the
    # roofline: MEASURED_PEAKS.json is the denominator; this shows what this
    # box moved today with a plain copy)
    stream = None
    if not sub:
        s_copy = session_copy_rate(torch, dev)
        stream = {"copy_GBps": round(s_copy, 1), "decode_kernel_vs_copy": round(achieved / s_copy, 4),
                  "method": "torch copy_ of 4 GiB bf16 buffers, read + write bytes, median of 20 runs, "
                            "CUDA events"}

    # ---- CPU baseline: the oracle on a bounded sample --------------------
    cpu = None
    if rank == 0 and ws == 1 and not sub and not args.no_cpu_baseline:
        per_step_pages = staged / K_ if K_ else 0.0
        cpu = cpu_baseline_leg(wl, dev, min(args.cpu_layers, wl.L), alpha, kv_bytes / K_, per_step_pages)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
            "steps": K_, "warmup": W_, "ms_per_step": round(ms_max / K_, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "fp8": "e4m3 KV, f16 MMA, fp32 accumulate",
                      "kivi2": "2-bit KV groups (fp16 scale/zero) + bf16 residual window, f16 MMA, "
                               "fp32 accumulate"}[args.kv_dtype],
            "data": "synthetic (seeded generator; recency-skewed K/V)",
            "config": {"workload": f"{wl.name}: {wl.nseq} seq x "
                                   f"{wl.prefill_lens[0] if wl.nseq == 1 else f'{min(wl.prefill_lens)}..{max(wl.prefill_lens)}'} "
                                   f"tokens (+1 per step), L={wl.L} Hq={wl.Hq} Hkv={wl.Hkv} d={wl.d}, 16-token pages"
                                   + (f", {wl.shared_prefix_tokens}-token shared prefix" if wl.shared_prefix_tokens else ""),
                       "global_batch": wl.nseq, "seq_len": max(wl.prefill_lens),
                       "alpha": alpha, "gather": gather,
                       "score_call": ("kvs_decode_step + kvs_score_update" if args.unfused else
                                      "kvs_decode_score_step: records scored in the decode epilogue "
                                      "(breakdown 'score' is then empty)"),
                       "select_call": ("KVS_GATHER_ASYNC: no host wait; counts read one step later"
                                       if gather in ("mirror", "ids") else "synchronising"),
                       **({"prefetch_budget": args.prefetch_budget} if gather == "prefetch" else {}),
                       **({"victims": args.victims} if gather in ("demote", "prefetch") else {}),
                       "l2": "inputs larger than L2 (KV per step >> 129 MB), no flush",
                       "parallelism": f"replicas x{ws}"},
            "decode_tok_per_s": round(tok_s, 2),
            "physical_bound": {
                "unique_kv_gbps": round(uniq_bytes / (ms / 1e3) / 1e9, 2),
                "logical_exceeds_measured_peak": bool(value > peak),
                "note": "logical bytes count a shared prefix once per sequence; unique bytes once"},
            "kv_gbps_pct_of_hbm": round(100 * value / peak, 2),
            "kv_gbps_pct_of_8tbs": round(100 * value / 8000.0, 2),
            "roofline": {"bound": "hbm", "kernel": "decode_kernel (split-K paged GQA)",
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": int(algo),
                         "avg_launch_ms": round(dec_avg, 4),
                         "launches_timed": f"{len(dec_steps)} of the {K_} timed steps (every {dec_every}th)",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback 6.8 TB/s"},
            "breakdown_ms": {k: round(v, 4) for k, v in part.items()},
            "scoring_overhead_pct": round(100 * (part["score"] + part["select_gather"]) /
                                          max(part["decode_step"], 1e-9), 2),
            "outside_decode_kernel_pct": round(100 * (ms_max / K_ - dec_avg) / dec_avg, 2),
            "gathered_pages_timed": staged,
            "demoted_and_readmitted_pages_timed": demoted,
            "demote_readmit_rounds": round_info,
            "prefetched_pages_timed": prefetched if gather == "prefetch" else None,
            "e2e": e2e,
            "literal_gather": literal,
            "cpu_baseline": cpu,
            "clocks": clk,
            "copy_rate_session": stream,
            "gpu_launches": launches,
            "wall_s_timed": round(wall, 3),
        }
        if sub:
            for k in ("literal_gather", "cpu_baseline", "copy_rate_session", "n_gpus", "metric", "unit",
                      "higher_is_better", "scaling", "vs_baseline", "data", "dtype"):
                line.pop(k, None)
        pipe.ctx.close()
        return line
    pipe.ctx.close()
    return None


def run_kvs(args):
    import torch
    from paged_kv_cache_flash_gb300 import build
    build.build()
    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    line = measure(args, args.workload, dev, ws, rank, local)
    if args.workload == "l70b_128k" and not args.no_batched:
        # the other workload the target names: the batched one, same steps,
        # warm-up and page format, its own line under "batched"
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        if hasattr(torch._C, "_host_emptyCache"):
            torch._C._host_emptyCache()     # the 128K run's pinned host mirror
        sub = measure(args, "l70b_batch16", dev, ws, rank, local, sub=True)
        if line is not None:
            line["batched"] = sub
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------- reference (oracle)


def run_reference(args):
    ws, rank, local = dist_info()
    if rank != 0:
        return
    import torch
    import workloads as W
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = W.workload(args.workload)
    layers = 1
    n = wl.prefill_lens[0] + 1
    q, Kc, Vc = cpu_sample(wl, n, layers, dev)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        time_oracle(wl, q, Kc, Vc, layers, threads)
    secs = [time_oracle(wl, q, Kc, Vc, layers, threads) for _ in range(args.steps)]
    sample_bytes = n * layers * wl.Hkv * wl.d * 2 * 2
    tot = sum(secs)
    value = sample_bytes * args.steps / tot / 1e9
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: 1 seq x {wl.prefill_lens[0]} tokens (oracle sample: "
                               f"layer 0 of {wl.L}, all {wl.Hq} heads, per step)",
                   "global_batch": 1, "seq_len": wl.prefill_lens[0]},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step: fp64 attention + block mass of layer 0 "
                                   f"({wl.Hq} heads x {n} tokens)"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvs(args)


if __name__ == "__main__":
    main()
