"""Benchmark of the head-aware paged attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama33_70b_prefill_128k|mistral7b_prefill_8k|llama3_8b_decode_32k]

Prints ONE JSON line (rank 0).  Default workload: the Llama-3.3-70B-shaped
long prefill, every one of its 64 layers (Hq 64 / Hkv 8, d 128, one
sequence of 131,072 tokens, page 64; 77 of the 512 (layer, KV head) units
GLOBAL by seed, the rest LOCAL(4, 8192)), each layer with its own policy
row and its own Q/K/V resident in HBM.  One step is one pass of the whole
path over that sequence: per layer the causal prefill of all 131,072 rows
and the trimmed KV write of the chunk (page allocation + scatter), then one
decode token per layer (append + split-KV decode), then the release of the
sequence's pages.  The head-class policy is set once, offline, before
timing.  The same line carries, under "decode", the Llama-3-8B-shaped
decode batch (32 layers, 32 sequences x 32,768 cached tokens, 64 steps).

Metric: visible-pair TFLOP/s (FLOP = 4 d per visible (query, key) pair, for
the prefill rows and the decode rows) for prefill workloads; visible-KV GB/s
(2 d bytes of K and V per visible key and head) for the decode workload.
The roofline of each record is its dominant kernel over all of its launches
in the timed steps (CUDA events around each launch on the launching stream).
Timing: CUDA events on the launching stream after W warm-up steps; L2 is
flushed (256 MB write) between steps, outside the timed events.  With
--gpus N > 1 (torchrun), every rank runs the same workload on its own GPU
(replicas; the path has no cross-GPU exchange) and the value is the sum of
the ranks' work over the slowest rank's time.

--impl reference times the CPU oracle (plain fp32 C, all host cores) on a
bounded sample of the same workload, in the same units, with the same config.
"""
from __future__ import annotations

import argparse
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

import workloads as W  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    QUERY = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and parts[1] != self.uuid:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[6 + k] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _dist_device():
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def reduce_max(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_dist_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units: float, ms: float, ws: int) -> float:
    """Whole-job rate: the units every rank processed, summed, over the
    slowest rank's time (units per second)."""
    if ws > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([units], dtype=torch.float64, device=_dist_device())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        units = float(t.item())
        ms = reduce_max(ms, ws)
    return units / (ms / 1e3)


# ------------------------------------------------------------ workloads

def unit_pages(p, n: int, P: int) -> int:
    """Pages one (sequence, layer, KV head) unit holds after n tokens (pool
    sizing only: GLOBAL ceil(n/P); LOCAL its sink pages plus at most its ring
    of ceil(W/P) + 1 pages; RETRIEVAL its listed positions below n)."""
    if p.kind == W.GLOBAL:
        return -(-n // P)
    if p.kind == W.LOCAL:
        ring = -(-p.window // P) + 1
        return -(-min(n, p.sink) // P) + min(ring, -(-max(0, n - p.sink) // P))
    return -(-int((np.asarray(p.idx) < n).sum()) // P)


class PrefillStep:
    """One sequence, every layer of the workload: per layer the causal
    prefill of the whole sequence as one chunk and the trimmed KV write of
    that chunk (page allocation + scatter); then one decode token in every
    layer (append + split-KV decode); then the release of the sequence's
    pages.  Each layer has its own head-class row and its own Q/K/V, all
    resident in HBM before timing; the policy is set once, offline."""

    def __init__(self, wl, device="cuda", layer_range=None):
        import torch
        from head_aware_paged_gb300 import Config, Policy, SegPagedCache
        self.wl = wl
        L = wl.seq_len
        self.L = L
        lo, hi = layer_range or (0, wl.layers)
        self.layer_ids = list(range(lo, hi))         # the workload's layers this step runs
        self.layers = hi - lo
        self.pols = W.policies(wl)[lo:hi]
        pages = sum(unit_pages(p, L + 1, wl.page) for row in self.pols for p in row)
        n_idx = sum(0 if p.idx is None else len(p.idx) for row in self.pols for p in row)
        self.cfg = Config(num_layers=self.layers, num_q_heads=wl.hq, num_kv_heads=wl.hkv,
                          head_dim=wl.d, page_size=wl.page, max_seqs=1, max_seq_len=L + 64,
                          num_pages=pages + 64, max_idx_per_seq=max(1, n_idx), max_tokens=L,
                          max_batch=1)
        self.cache = SegPagedCache(self.cfg)
        self.cache.set_policy(0, [[Policy(p.kind, p.sink, p.window,
                                          None if p.idx is None else p.idx.tolist())
                                   for p in row] for row in self.pols])
        # per layer: rows 0..L-1 are the prefill chunk, row L the decode token
        self.q, self.k, self.v, self.q1, self.k1, self.v1 = [], [], [], [], [], []
        for l in self.layer_ids:
            q, k, v = W.qkv(wl, L + 1, 0, l, device=device)
            for lst, t in ((self.q, q), (self.k, k), (self.v, v)):
                lst.append(t[:L])
            for lst, t in ((self.q1, q), (self.k1, k), (self.v1, v)):
                lst.append(t[L:])
            del q, k, v
        self.out = torch.empty_like(self.q[0])
        self.lse = torch.empty(L, wl.hq, dtype=torch.float32, device=device)
        self.out1 = torch.empty_like(self.q1[0])
        self.lse1 = torch.empty(1, wl.hq, dtype=torch.float32, device=device)
        grp = wl.hq // wl.hkv
        self.pf_flop = [4 * wl.d * self.cache.count_prefill_pairs(0, l, 0, L)
                        for l in range(self.layers)]
        dec_pairs = sum(self.cache.count_decode_bytes(l, [0], [L]) // (2 * wl.d * 2) * grp
                        for l in range(self.layers))
        self.prefill_flop = sum(self.pf_flop)
        self.work = self.prefill_flop + 4 * wl.d * dec_pairs      # FLOP per step
        # launches per step: per layer the prefill (plus the copy kernel of a
        # work list too large for the kernel parameters) and the chunk's
        # append (allocator + scatter); per layer the decode token's append
        # and decode; one release
        pairs = grp // 2 if grp % 2 == 0 else grp
        items = wl.hkv * (-(-L // 128)) * pairs
        words = items + (min(items, 152) + 1 + 3) // 4
        pf_launches = 1 + (0 if words <= 1344 else 1)
        self.kernels_per_step = self.layers * (pf_launches + 2) + self.layers * 3 + 1
        self.unit = "TFLOP/s"

    def run(self, ev_pf=None):
        """One step; ev_pf (optional): a (start, end) event pair per layer
        that the library records right before and after that layer's
        prefill kernels (host planning outside the interval)."""
        c = self.cache
        for l in range(self.layers):
            if ev_pf is not None:
                c.set_launch_events(*ev_pf[l])
            c.prefill(l, [0], [0, self.L], self.q[l], self.k[l], self.v[l], self.out, self.lse)
            c.append_kv(l, [0], [0, self.L], self.k[l], self.v[l])
        for l in range(self.layers):
            c.append_kv(l, [0], [0, 1], self.k1[l], self.v1[l])
            c.decode(l, [0], self.q1[l], self.out1, self.lse1)
        c.release(0)

    # host-buffer (end-to-end) variant: every layer's q/k/v chunk is uploaded
    # from pinned host memory and its out/lse read back; the decode tokens of
    # all layers go up in one packed copy and their outputs come back in one.
    # Layers alternate between two device buffer sets and run on upload,
    # kernel and download streams, so layer l+1's upload and layer l-1's
    # download overlap layer l's kernels.  One pinned host set of chunk
    # inputs (layer 0's values) is uploaded for every layer: the bytes moved
    # are those of a real pass, only the values repeat.
    def setup_e2e(self):
        import torch
        pin = lambda t: t.cpu().pin_memory()
        self.h_in = [pin(t) for t in (self.q[0], self.k[0], self.v[0])]
        self.dset = [[torch.empty_like(t) for t in (self.q[0], self.k[0], self.v[0], self.out, self.lse)]
                     for _ in range(2)]
        self.h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (self.out, self.lse)]
                      for _ in range(2)]
        nq, nk = self.q1[0].numel(), self.k1[0].numel()
        self.tok_split = (nq, nq + nk, nq + 2 * nk)
        tok = torch.cat([torch.cat([self.q1[l].reshape(-1), self.k1[l].reshape(-1), self.v1[l].reshape(-1)])
                         for l in range(self.layers)])
        self.tok_words = nq + 2 * nk
        self.h_tok = tok.cpu().pin_memory()
        self.d_tok = torch.empty_like(tok)
        no, nl = self.out1.numel(), self.lse1.numel()    # out bf16, lse fp32 (2 bf16 slots each)
        self.tokout_words = no + 2 * nl
        self.d_tokout = torch.empty(self.tokout_words * self.layers, dtype=torch.bfloat16, device=tok.device)
        self.h_tokout = torch.empty(self.d_tokout.numel(), dtype=torch.bfloat16).pin_memory()
        self.streams = [torch.cuda.Stream() for _ in range(3)]        # upload, kernels, download
        self.ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}
        self.ev_tok = {k: torch.cuda.Event() for k in ("in", "done", "out")}
        self.h2d_bytes = (self.layers * sum(t.numel() * t.element_size() for t in self.h_in)
                          + self.h_tok.numel() * 2)
        self.d2h_bytes = (self.layers * sum(t.numel() * t.element_size() for t in self.h_out[0])
                          + self.h_tokout.numel() * 2)

    def run_e2e_steps(self, n):
        """n steps through the C ABI with host buffers; returns CUDA events
        around all of them (first upload to last download)."""
        import torch
        sh, sc, sd = self.streams
        cur = torch.cuda.current_stream()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(cur)
        for st_ in self.streams:
            st_.wait_event(start)
        c = self.cache
        a, b_, e_ = self.tok_split
        no, wi, wo = self.out1.numel(), self.tok_words, self.tokout_words
        g = 0
        for step in range(n):
            with torch.cuda.stream(sh):
                if step >= 1:
                    sh.wait_event(self.ev_tok["done"])          # last step's tokens are read
                self.d_tok.copy_(self.h_tok, non_blocking=True)
                self.ev_tok["in"].record(sh)
            for l in range(self.layers):
                b = g % 2
                q, k, v, out, lse = self.dset[b]
                with torch.cuda.stream(sh):
                    if g >= 2:
                        sh.wait_event(self.ev["done"][b])      # layer g-2 has read these inputs
                    for d, h in zip((q, k, v), self.h_in):
                        d.copy_(h, non_blocking=True)
                    self.ev["in"][b].record(sh)
                sc.wait_event(self.ev["in"][b])
                if g >= 2:
                    sc.wait_event(self.ev["out"][b])           # layer g-2's outputs are home
                c.prefill(l, [0], [0, self.L], q, k, v, out, lse, stream=sc)
                c.append_kv(l, [0], [0, self.L], k, v, stream=sc)
                self.ev["done"][b].record(sc)
                sd.wait_event(self.ev["done"][b])
                with torch.cuda.stream(sd):
                    for h, d in zip(self.h_out[b], (out, lse)):
                        h.copy_(d, non_blocking=True)
                    self.ev["out"][b].record(sd)
                g += 1
            sc.wait_event(self.ev_tok["in"])
            if step >= 1:
                sc.wait_event(self.ev_tok["out"])               # last step's token outputs are home
            for l in range(self.layers):
                ti, to = self.d_tok[l * wi:(l + 1) * wi], self.d_tokout[l * wo:(l + 1) * wo]
                c.append_kv(l, [0], [0, 1], ti[a:b_].view(self.k1[0].shape),
                            ti[b_:e_].view(self.v1[0].shape), stream=sc)
                c.decode(l, [0], ti[:a].view(self.q1[0].shape), to[:no].view(self.out1.shape),
                         to[no:].view(torch.float32).view(self.lse1.shape), stream=sc)
            c.release(0, stream=sc)
            self.ev_tok["done"].record(sc)
            sd.wait_event(self.ev_tok["done"])
            with torch.cuda.stream(sd):
                self.h_tokout.copy_(self.d_tokout, non_blocking=True)
                self.ev_tok["out"].record(sd)
        for st_ in self.streams:
            cur.wait_stream(st_)
        end.record(cur)
        return start, end

    def free_e2e(self):
        for name in ("h_in", "dset", "h_out", "h_tok", "d_tok", "d_tokout", "h_tokout"):
            if hasattr(self, name):
                delattr(self, name)

    def oracle_rows(self, layer, rows, threads):
        """The fp32 C oracle on the given query rows (all heads) of one layer;
        returns (seconds, visible-pair FLOP)."""
        import oracle
        from oracle import accounting
        pt = [(p.kind, p.sink, p.window, None if p.idx is None else p.idx.tolist())
              for p in self.pols[layer]]
        qf = self.q[layer][rows].float().cpu().numpy()
        kf = self.k[layer].float().cpu().numpy()
        vf = self.v[layer].float().cpu().numpy()
        t0 = time.perf_counter()
        oracle.attend(qf, kf, vf, rows, pt, "f32", threads=threads)
        dt = time.perf_counter() - t0
        grp = self.wl.hq // self.wl.hkv
        pairs = sum(grp * int(accounting.vis_count_closed(p[0], p[1], p[2], p[3], rows).sum()) for p in pt)
        return dt, 4 * self.wl.d * pairs


FP8_SCALE = 5.6 / 448.0


class DecodeStep:
    """Llama-3-8B-shaped decode: per layer, append one token per sequence and
    decode the batch; one step = all layers."""

    def __init__(self, wl, device="cuda", layers=None, fp8=False):
        import torch
        from head_aware_paged_gb300 import KV_BF16, KV_FP8, Config, Policy, SegPagedCache
        self.wl = wl
        self.fp8 = fp8
        self.layers = layers or wl.layers
        B, n = wl.seqs, wl.seq_len
        pols = W.policies(wl)[:self.layers]
        self.pols = pols
        steps_cap = 256
        pages = 0
        for row in pols:
            for p in row:
                if p.kind == W.GLOBAL:
                    pages += B * ((n + steps_cap) // wl.page + 1)
                else:
                    pages += B * ((p.sink + wl.page - 1) // wl.page + (p.window + wl.page - 1) // wl.page + 1)
        self.cfg = Config(num_layers=self.layers, num_q_heads=wl.hq, num_kv_heads=wl.hkv,
                          head_dim=wl.d, page_size=wl.page, max_seqs=B, max_seq_len=n + steps_cap,
                          num_pages=pages + 16, max_tokens=max(n, B), max_batch=B,
                          kv_dtype=KV_FP8 if fp8 else KV_BF16)
        self.cache = SegPagedCache(self.cfg)
        if fp8:     # one scale for every channel: |x| up to 5.6 (N(0,1) data) maps inside +-448
            sc = np.full((wl.hkv, wl.d), FP8_SCALE, np.float32)
            for l in range(self.layers):
                self.cache.set_kv_scales(l, sc, sc)
        cp = [[Policy(p.kind, p.sink, p.window) for p in row] for row in pols]
        for b in range(B):
            self.cache.set_policy(b, cp)
        for l in range(self.layers):
            for b in range(B):
                k = W.normal((n, wl.hkv, wl.d), W.tensor_seed(0, "k", b, l), device=device)
                v = W.normal((n, wl.hkv, wl.d), W.tensor_seed(0, "v", b, l), device=device)
                self.cache.build(b, l, k, v)
                del k, v
        torch.cuda.synchronize()
        self.B, self.n = B, n
        self.qs = W.normal((B, wl.hq, wl.d), 11, device=device)
        self.kn = W.normal((B, wl.hkv, wl.d), 12, device=device)
        self.vn = W.normal((B, wl.hkv, wl.d), 13, device=device)
        self.out = torch.empty_like(self.qs)
        self.lse = torch.empty(B, wl.hq, dtype=torch.float32, device=device)
        self.cu = list(range(B + 1))
        self.seqs = list(range(B))
        self.unit = "GB/s"
        self.kernels_per_step = 3 * self.layers
        self.t = n      # position of the next token

    def step_bytes(self, t):
        return sum(self.cache.count_decode_bytes(l, self.seqs, [t] * self.B)
                   for l in range(self.layers))

    # host-buffer (end-to-end) variant: a step's q / new k / new v for all
    # layers come from pinned host memory in one packed copy and its out /
    # lse for all layers go back in one; two steps are in flight (two device
    # buffer sets) on upload, kernel and download streams, so step i+1's
    # upload and step i-1's download overlap step i's kernels
    def setup_e2e(self):
        import torch
        nq, nk = self.qs.numel(), self.kn.numel()
        self.e2e_split = (nq, nq + nk, nq + 2 * nk)
        per_layer = torch.cat([self.qs.reshape(-1), self.kn.reshape(-1), self.vn.reshape(-1)])
        self.e2e_in_words = per_layer.numel()
        self.h_in = per_layer.repeat(self.layers).cpu().pin_memory()
        no, nl = self.out.numel(), self.lse.numel()      # out bf16, lse fp32 (2 bf16 slots each)
        self.e2e_out_words = no + 2 * nl
        dev = per_layer.device
        self.d_in = [torch.empty(self.h_in.numel(), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.d_out = [torch.empty(self.e2e_out_words * self.layers, dtype=torch.bfloat16, device=dev)
                      for _ in range(2)]
        self.h_out = [torch.empty(self.e2e_out_words * self.layers, dtype=torch.bfloat16).pin_memory()
                      for _ in range(2)]
        self.streams = [torch.cuda.Stream() for _ in range(3)]
        self.ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}
        self.h2d_bytes = self.h_in.numel() * 2
        self.d2h_bytes = self.h_out[0].numel() * 2

    def run_e2e_steps(self, n):
        """n decode steps through the C ABI with host buffers; returns (CUDA
        events around all of them, visible bytes they read)."""
        import torch
        sh, sc, sd = self.streams
        cur = torch.cuda.current_stream()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(cur)
        for st_ in self.streams:
            st_.wait_event(start)
        a, b, e = self.e2e_split
        no, wi, wo = self.out.numel(), self.e2e_in_words, self.e2e_out_words
        work = 0
        for step in range(n):
            work += self.step_bytes(self.t)
            k = step % 2
            din, dout = self.d_in[k], self.d_out[k]
            with torch.cuda.stream(sh):
                if step >= 2:
                    sh.wait_event(self.ev["done"][k])        # step-2's kernels read din
                din.copy_(self.h_in, non_blocking=True)
                self.ev["in"][k].record(sh)
            sc.wait_event(self.ev["in"][k])
            if step >= 2:
                sc.wait_event(self.ev["out"][k])            # step-2's outputs are home
            for l in range(self.layers):
                li, lo_ = din[l * wi:(l + 1) * wi], dout[l * wo:(l + 1) * wo]
                self.cache.append_kv(l, self.seqs, self.cu, li[a:b].view(self.kn.shape),
                                     li[b:e].view(self.vn.shape), stream=sc)
                self.cache.decode(l, self.seqs, li[:a].view(self.qs.shape), lo_[:no].view(self.out.shape),
                                  lo_[no:].view(torch.float32).view(self.lse.shape), stream=sc)
            self.ev["done"][k].record(sc)
            sd.wait_event(self.ev["done"][k])
            with torch.cuda.stream(sd):
                self.h_out[k].copy_(dout, non_blocking=True)
                self.ev["out"][k].record(sd)
            self.t += 1
        for st_ in self.streams:
            cur.wait_stream(st_)
        end.record(cur)
        return start, end, work

    def run(self, ev_pf=None):
        """One step; ev_pf (optional): a (start, end) event pair per layer
        that the library records right before and after that layer's
        decode kernel (host planning outside the interval)."""
        c = self.cache
        for l in range(self.layers):
            c.append_kv(l, self.seqs, self.cu, self.kn, self.vn)
            if ev_pf is not None:
                c.set_launch_events(*ev_pf[l])
            c.decode(l, self.seqs, self.qs, self.out, self.lse)
        self.t += 1


# ---------------------------------------------------------------- traffic

def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 3 and not line.startswith("#") and parts[0] == kernel + "/" + workload:
                    return int(parts[2]) if parts[1] == source_sha() else None
    except OSError:
        pass
    return None


def bench_layer(wl) -> int:
    """The layer --op chunk_prefill runs: the first whose policy has a GLOBAL
    KV head (it carries the full-causal work), else layer 0."""
    pols = W.policies(wl)
    return next((l for l, row in enumerate(pols) if any(p.kind == W.GLOBAL for p in row)), 0)


def source_sha():
    import hashlib
    h = hashlib.sha1()
    cs = os.path.join(ROOT, "head_aware_paged_gb300", "csrc")
    for f in sorted(os.listdir(cs)):
        with open(os.path.join(cs, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


METRIC = "SegPaged prefill TFLOP/s & decode visible-KV GB/s, % of GB300 roofline"
DATA = "synthetic (seeded N(0,1), pages' shapes)"
DECODE_WL = "llama3_8b_decode_32k"


def is_decode(wl) -> bool:
    return wl.decode_steps > 0 and wl.name.startswith("llama3_8b")


def gpu_uuid():
    import torch
    try:
        u = str(torch.cuda.get_device_properties(0).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- main arms

def timed_steps(st, steps, warmup, ws, rank, decode):
    """warmup untimed steps, then `steps` timed ones bracketed by a barrier
    and a synchronize; L2 is flushed before each step outside its events.
    Returns the step times, the dominant kernel's summed launch times per
    step, the work per step (and of those launches) and the clock record."""
    import torch
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(warmup):
        st.run()
    torch.cuda.synchronize()
    assert st.cache.status() == 0
    E = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(E(), E()) for _ in range(steps)]
    evk = [[(E(), E()) for _ in range(st.layers)] for _ in range(steps)]
    for row in evk:                 # the library records these: create them first
        for pair in row:
            for e in pair:
                e.record()
    torch.cuda.synchronize()
    work, kern_work = [], []
    clocks = ClockSampler(gpu_uuid() if rank == 0 else None)
    if rank == 0:
        clocks.start()
        time.sleep(0.4)
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(steps):
        flush.random_(0, 255) if i == 0 else flush.fill_(i & 0xFF)
        if decode:
            work.append(st.step_bytes(st.t))
            kern_work.append(work[-1])                   # every layer's decode launch
        else:
            work.append(st.work)
            kern_work.append(st.prefill_flop)             # every layer's prefill launch
        ev[i][0].record(stream)
        st.run(evk[i])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if rank == 0 else None
    assert st.cache.status() == 0
    del flush
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [sum(a.elapsed_time(b) for a, b in row) for row in evk]
    return step_ms, kern_ms, work, kern_work, clk


def prefill_record(args, wl, ws, rank, steps):
    import torch
    st = PrefillStep(wl, layer_range=layer_range(args, wl))
    torch.cuda.synchronize()
    step_ms, kern_ms, work, kern_work, clk = timed_steps(st, steps, args.warmup, ws, rank, False)
    total_ms = reduce_max(float(sum(step_ms)), ws)
    value = job_rate(float(sum(work)), float(sum(step_ms)), ws) * 1e-12
    # end to end through the same C-ABI calls with host buffers
    e2e = None
    if not args.no_e2e:
        st.setup_e2e()
        st.run_e2e_steps(1)
        torch.cuda.synchronize()
        e2e_steps = 3 if st.layers > 1 else max(3, min(steps, 10))
        barrier(ws)
        e0, e1 = st.run_e2e_steps(e2e_steps)
        torch.cuda.synchronize()
        assert st.cache.status() == 0
        e2e = {"value": job_rate(float(st.work * e2e_steps), e0.elapsed_time(e1), ws) * 1e-12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": st.h2d_bytes,
               "d2h_bytes_per_step": st.d2h_bytes, "steps": e2e_steps}
        st.free_e2e()
    rec = None
    if rank == 0:
        peaks, src = load_peaks()
        launch_ms = float(np.sum(kern_ms)) / (steps * st.layers)
        achieved = float(np.sum(kern_work)) / (float(np.sum(kern_ms)) / 1e3) / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": load_traffic("k_prefill", wl.name),
                "kernel": "k_prefill", "peak_source": src + " bf16_tflops (burst)",
                "launches_per_step": st.layers,
                "algorithmic_flop_per_launch": st.prefill_flop / st.layers,
                "avg_launch_ms": launch_ms}
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            cpu = prefill_cpu_baseline(st)
        rec = {"value": value, "unit": "TFLOP/s", "steps": steps, "ms_per_step": total_ms / steps,
               "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": st.kernels_per_step * steps, "clocks": clk}
    st.cache.close()
    del st
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    return rec


def decode_record(args, wl, ws, rank, steps):
    import torch
    fp8 = args.kv_dtype == "fp8"
    st = DecodeStep(wl, layers=args.decode_layers or None, fp8=fp8)
    step_ms, kern_ms, work, kern_work, clk = timed_steps(st, steps, args.warmup, ws, rank, True)
    total_ms = reduce_max(float(sum(step_ms)), ws)
    value = job_rate(float(sum(work)), float(sum(step_ms)), ws) * 1e-9
    e2e = None
    if not args.no_e2e:
        st.setup_e2e()
        st.run_e2e_steps(1)
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1, w = st.run_e2e_steps(3)
        torch.cuda.synchronize()
        assert st.cache.status() == 0
        e2e = {"value": job_rate(float(w), e0.elapsed_time(e1), ws) * 1e-9, "unit": "GB/s",
               "h2d_bytes_per_step": st.h2d_bytes, "d2h_bytes_per_step": st.d2h_bytes, "steps": 3}
    rec = None
    if rank == 0:
        peaks, src = load_peaks()
        achieved = float(np.sum(kern_work)) / (float(np.sum(kern_ms)) / 1e3) / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": load_traffic("k_decode", wl.name + ("_fp8" if fp8 else "")),
                "kernel": "k_decode", "peak_source": src + " hbm_gbs",
                "launches_per_step": st.layers,
                "algorithmic_bytes_per_launch": float(np.mean(kern_work)) / st.layers,
                "avg_launch_ms": float(np.sum(kern_ms)) / (steps * st.layers)}
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            cpu = decode_cpu_baseline(st, wl)
        rec = {"value": value, "unit": "GB/s", "steps": steps, "warmup": args.warmup,
               "ms_per_step": total_ms / steps,
               "dtype": "e4m3 K/V pages, f16 MMA" if fp8 else "bf16",
               "config": config_dict(wl, args),
               "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": st.kernels_per_step * steps, "clocks": clk}
    st.cache.close()
    del st
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, ws, rank):
    import torch
    from head_aware_paged_gb300 import build as _b
    if rank == 0:
        _b.build()
    barrier(ws)
    torch.cuda.init()
    wl = W.WORKLOADS[args.workload]
    decode = is_decode(wl)
    if args.kv_dtype == "fp8" and not decode:
        raise SystemExit("--kv-dtype fp8 applies to the decode workload and --op chunk_prefill "
                         "(the prefill step has no cached history)")
    steps = args.steps
    if decode:
        rec = decode_record(args, wl, ws, rank, steps)
    else:
        rec = prefill_record(args, wl, ws, rank, steps)
        if wl.layers > 1 and not args.no_decode_record:
            # the decode half of the metric: the Llama-3-8B-shaped decode
            # batch at its configuration's 64 steps
            drec = decode_record(args, W.WORKLOADS[DECODE_WL], ws, rank, 64)
            if rank == 0:
                drec["workload"] = DECODE_WL
                drec["metric"] = "decode visible-KV GB/s"
                rec["decode"] = drec
            # the same batch over FP8 (e4m3) pages, bytes counted as stored
            fargs = argparse.Namespace(**vars(args))
            fargs.kv_dtype, fargs.no_cpu_baseline = "fp8", True
            frec = decode_record(fargs, W.WORKLOADS[DECODE_WL], ws, rank, 64)
            if rank == 0:
                frec["workload"] = DECODE_WL
                frec["metric"] = "decode visible-KV GB/s (FP8 pages)"
                rec["decode_fp8"] = frec
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": rec.pop("value"), "unit": rec.pop("unit"), "n_gpus": ws,
            "steps": rec.pop("steps"), "warmup": args.warmup, "ms_per_step": rec.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": rec.pop("dtype", "bf16"), "data": DATA, "config": rec.pop("config", None)
            or config_dict(wl, args)}
    line.update(rec)
    return line


def layer_range(args, wl):
    """--layers: all of the workload's layers (default), the first N ("N") or
    layers a .. b-1 ("a:b")."""
    if not args.layers:
        return (0, wl.layers)
    if ":" in args.layers:
        a, b = (int(x) for x in args.layers.split(":"))
    else:
        a, b = 0, int(args.layers)
    if not 0 <= a < b <= wl.layers:
        raise SystemExit("--layers must select layers inside 0 .. %d" % (wl.layers - 1))
    return (a, b)


def config_dict(wl, args):
    """The workload as the line names it (the reference arm prints the same)."""
    d = {"workload": wl.name, "layers": wl.layers, "hq": wl.hq, "hkv": wl.hkv, "head_dim": wl.d,
         "page_size": wl.page, "local": [wl.local_sink, wl.local_window],
         "global_units": wl.n_global,
         "l2": "flushed between steps (256 MB write outside the timed events)",
         "parallelism": "replicas (no cross-GPU exchange on this path)"}
    if is_decode(wl):
        fp8 = args.kv_dtype == "fp8"
        d.update({"layers": args.decode_layers or wl.layers, "batch": wl.seqs,
                  "cached_tokens": wl.seq_len,
                  "step": "all layers: append 1 token/seq + split-KV decode",
                  "kv_dtype": "fp8_e4m3" if fp8 else "bf16"})
        if fp8:
            d["workload"] = wl.name + "_fp8"
            d["kv_scales"] = "%.6g for every channel of K and V" % FP8_SCALE
    else:
        lo, hi = layer_range(args, wl)
        if (lo, hi) != (0, wl.layers):
            d["layers"] = hi - lo
            d["layer_range"] = [lo, hi]
        d.update({"seq_len": wl.seq_len, "batch": wl.seqs,
                  "step": "every layer: prefill of the whole sequence + trimmed KV write; then 1 "
                          "decode token per layer (append + decode); release"})
    return d


def prefill_cpu_baseline(st, target_s=12.0, rows_per_head=256):
    """The fp32 C oracle on all host cores: 256 sampled query rows (every
    query head) per layer, layer after layer until about target_s seconds of
    oracle time; plus a smaller sample on one thread."""
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(5)
    n = min(rows_per_head, st.L)
    busy = flop = 0.0
    done = []
    for l in range(st.layers):
        rows = np.sort(rng.choice(st.L, size=n, replace=False))
        dt, fl = st.oracle_rows(l, rows, threads)
        busy += dt
        flop += fl
        done.append(l)
        if busy >= target_s:
            break
    rows1 = np.sort(rng.choice(st.L, size=max(4, n // 64), replace=False))
    dt1, fl1 = st.oracle_rows(0, rows1, 1)
    return {"value": flop / busy / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d sampled query rows of every query head on %d of %d layers (layers %d-%d), "
                      "fp32 C oracle" % (n, len(done), st.layers, done[0], done[-1]),
            "one_thread": {"value": fl1 / dt1 / 1e12, "cores": 1,
                           "sample": "%d query rows of layer 0 (all %d heads)" % (len(rows1), st.wl.hq)}}


def decode_cpu_baseline(st, wl):
    import oracle
    threads = os.cpu_count() or 1
    # layer 0 of two sequences, one decode query each, K/V regenerated on the host
    seqs = [0, wl.seqs - 1]
    busy = 0.0
    nbytes = 0
    pt = [(p.kind, p.sink, p.window, None) for p in st.pols[0]]
    qf = st.qs.float().cpu().numpy()
    t = st.n - 1
    k0 = v0 = None
    for b in seqs:
        k = W.normal((st.n, wl.hkv, wl.d), W.tensor_seed(0, "k", b, 0)).float().numpy()
        v = W.normal((st.n, wl.hkv, wl.d), W.tensor_seed(0, "v", b, 0)).float().numpy()
        if b == 0:
            k0, v0 = k, v
        t1 = time.perf_counter()
        oracle.attend(qf[b:b + 1], k, v, [t], pt, "f32", threads=threads)
        busy += time.perf_counter() - t1
        nbytes += st.cache.count_decode_bytes(0, [b], [t])
    # the same query of sequence 0 on one thread
    t1 = time.perf_counter()
    oracle.attend(qf[0:1], k0, v0, [t], pt, "f32", threads=1)
    one = {"value": st.cache.count_decode_bytes(0, [0], [t]) / (time.perf_counter() - t1) / 1e9,
           "cores": 1, "sample": "layer 0, sequence 0, one decode query"}
    return {"value": nbytes / busy / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "layer 0, sequences 0 and %d, one decode query each over %d cached "
                      "tokens (fp32 C oracle)" % (wl.seqs - 1, st.n), "one_thread": one}


def reference_steps(args, one, unit, scale):
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    work = 0
    for _ in range(args.steps):
        work += one()
    dt = time.perf_counter() - t0
    return work * scale / dt, dt


def reference_decode(args, wl, threads, steps=None):
    """The oracle on one decode query (all heads) of one Llama-3-8B-shaped
    sequence of 32,768 cached tokens, layer 0, per step."""
    import oracle
    from oracle import accounting
    L = wl.seq_len
    pt = [(p.kind, p.sink, p.window, None) for p in W.policies(wl)[0]]
    k = W.normal((L, wl.hkv, wl.d), W.tensor_seed(0, "k", 0, 0)).float().numpy()
    v = W.normal((L, wl.hkv, wl.d), W.tensor_seed(0, "v", 0, 0)).float().numpy()
    q = W.normal((1, wl.hq, wl.d), 11).float().numpy()
    nb = sum(int(accounting.vis_count_closed(p[0], p[1], p[2], p[3], np.array([L - 1]))[0])
             for p in pt) * 2 * wl.d * 2

    def one():
        oracle.attend(q, k, v, [L - 1], pt, "f32", threads=threads)
        return nb
    a = argparse.Namespace(**vars(args))
    if steps is not None:
        a.steps = steps
    value, dt = reference_steps(a, one, "GB/s", 1e-9)
    return value, dt / a.steps * 1e3, a.steps, "one decode query of one sequence, layer 0, fp32 C oracle"


def run_reference(args, ws, rank):
    """The CPU oracle as the reference arm: each step one bounded sample of
    the same workload, in the same units."""
    if ws > 1 and rank != 0:
        return None
    import oracle
    from oracle import accounting
    wl = W.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(1)
    extra = {}
    if is_decode(wl):
        value, ms, steps, sample = reference_decode(args, wl, threads)
        unit = "GB/s"
    else:
        L = wl.seq_len
        pols = W.policies(wl)
        # up to two layers' K/V on the host (the first with a GLOBAL head and
        # the next), drawn from the workload's seeds; query rows sampled per step
        l0 = bench_layer(wl)
        layers = sorted({l0, (l0 + 1) % wl.layers})
        kv = {}
        for l in layers:
            kv[l] = (W.normal((L, wl.hkv, wl.d), W.tensor_seed(0, "k", 0, l), wl.k_scale).float().numpy(),
                     W.normal((L, wl.hkv, wl.d), W.tensor_seed(0, "v", 0, l)).float().numpy())
        grp = wl.hq // wl.hkv
        nrows = 48
        state = {"i": 0}

        def one():
            l = layers[state["i"] % len(layers)]
            state["i"] += 1
            pt = [(p.kind, p.sink, p.window, None if p.idx is None else p.idx.tolist()) for p in pols[l]]
            rows = np.sort(rng.choice(L, size=nrows, replace=False))
            q = W.normal((nrows, wl.hq, wl.d), W.tensor_seed(0, "q", 0, l, state["i"])).float().numpy()
            oracle.attend(q, kv[l][0], kv[l][1], rows, pt, "f32", threads=threads)
            return 4 * wl.d * sum(grp * int(accounting.vis_count_closed(p[0], p[1], p[2], p[3], rows).sum())
                                  for p in pt)
        value, dt = reference_steps(args, one, "TFLOP/s", 1e-12)
        ms, steps, unit = dt / args.steps * 1e3, args.steps, "TFLOP/s"
        sample = "%d random query rows (all heads) per step of layer %s, fp32 C oracle" % (
            nrows, " / ".join(str(l) for l in layers))
        if wl.layers > 1 and not args.no_decode_record:
            dwl = W.WORKLOADS[DECODE_WL]
            dv, dms, dsteps, dsample = reference_decode(args, dwl, threads, steps=3)
            extra["decode"] = {"workload": DECODE_WL, "metric": "decode visible-KV GB/s", "value": dv,
                               "unit": "GB/s", "steps": dsteps, "ms_per_step": dms,
                               "config": config_dict(dwl, args),
                               "cpu_baseline": {"value": dv, "unit": "GB/s", "kind": "oracle",
                                                "cores": threads, "sample": dsample},
                               "e2e": {"value": dv, "unit": "GB/s", "h2d_bytes_per_step": 0,
                                       "d2h_bytes_per_step": 0}}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": ws,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": DATA,
            "config": config_dict(wl, args),
            "cpu_baseline": {"value": value, "unit": unit, "kind": "oracle", "cores": threads,
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    line.update(extra)
    return line


def stored_rows(pols_row, n: int, seqs: int, page: int) -> int:
    """K rows one layer stores for `seqs` sequences of n tokens (page rules:
    GLOBAL n, LOCAL sink + its ring of ceil(W / P) + 1 pages, RETRIEVAL the
    listed positions below n)."""
    rows = 0
    for p in pols_row:
        if p.kind == W.GLOBAL:
            rows += n
        elif p.kind == W.LOCAL:
            ring = (-(-p.window // page) + 1) * page
            rows += min(n, p.sink) + min(max(n - p.sink, 0), ring)
        else:
            rows += int((np.asarray(p.idx) < n).sum())
    return rows * seqs


def run_op_rope(args):
    """sp_rope_realign over every stored K row of one layer of the
    Llama-3-8B-shaped decode batch (32 sequences x 32,768 tokens): HBM-bound,
    2 * 2d bytes per rotated row (read + write)."""
    import torch
    wl = W.WORKLOADS["llama3_8b_decode_32k"]
    fp8 = args.kv_dtype == "fp8"
    st = DecodeStep(wl, layers=1, fp8=fp8)
    c = st.cache
    nbytes = stored_rows(st.pols[0], st.n, st.B, wl.page) * 2 * wl.d * (1 if fp8 else 2)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        c.rope_realign(0, st.seqs, 1000)
    torch.cuda.synchronize()
    peaks, src = load_peaks()
    props = torch.cuda.get_device_properties(0)
    u = str(getattr(props, "uuid", ""))
    clocks = ClockSampler(u if u.startswith("GPU-") else ("GPU-" + u if u else None))
    clocks.start()
    time.sleep(0.4)
    ms = []
    for _ in range(args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        c.rope_realign(0, st.seqs, 1000)
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    clk = clocks.stop()
    assert c.status() == 0
    total = sum(ms)
    gbs = nbytes * args.steps / (total / 1e3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"metric": "RoPE realignment of stored K rows, GB/s moved (read + write)",
            "op": "rope_realign", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps, "higher_is_better": True,
            "dtype": "e4m3 K pages (fp32 rotation)" if fp8 else "bf16",
            "data": "synthetic (seeded N(0,1), pages' shapes)",
            "config": {"workload": "llama3_8b_decode_32k%s, layer 0, all 32 sequences" % ("_fp8" if fp8 else ""),
                       "bytes_per_call": nbytes, "l2": "flushed between calls"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": None, "kernel": "k_rope",
                         "peak_source": "%s hbm_gbs" % src},
            "clocks": clk}


def run_op_chunk(args):
    """Chunked prefill over cached history: the Mistral-7B-shaped layer's
    policies, 8,192 tokens already in the cache (bf16 or FP8 pages), then a
    2,048-row chunk prefilled over them (CUDA events around the call; the
    chunk is re-run on the same history each step)."""
    import torch
    from head_aware_paged_gb300 import KV_BF16, KV_FP8, Config, Policy, SegPagedCache
    wl = W.WORKLOADS["mistral7b_prefill_8k"]
    fp8 = args.kv_dtype == "fp8"
    layer = bench_layer(wl)
    row = W.policies(wl)[layer]
    H, C = 8192, 2048
    pol = [[Policy(p.kind, p.sink, p.window, None if p.idx is None else p.idx.tolist()) for p in row]]
    pages = len(row) * ((H + C) // wl.page + 4)
    cache = SegPagedCache(Config(num_layers=1, num_q_heads=wl.hq, num_kv_heads=wl.hkv, head_dim=wl.d,
                                 page_size=wl.page, max_seqs=1, max_seq_len=H + C + 64, num_pages=pages,
                                 max_idx_per_seq=max(1, sum(0 if p.idx is None else len(p.idx) for p in row)),
                                 max_tokens=H + C, max_batch=1, kv_dtype=KV_FP8 if fp8 else KV_BF16))
    cache.set_policy(0, pol)
    q, k, v = W.qkv(wl, H + C, 0, 0, device="cuda")
    if fp8:
        sc = np.full((wl.hkv, wl.d), FP8_SCALE, np.float32)
        cache.set_kv_scales(0, sc, sc)
    cache.build(0, 0, k[:H].contiguous(), v[:H].contiguous())
    qc, kc, vc = q[H:].contiguous(), k[H:].contiguous(), v[H:].contiguous()
    out = torch.empty_like(qc)
    lse = torch.empty(C, wl.hq, dtype=torch.float32, device="cuda")
    flop = 4 * wl.d * cache.count_prefill_pairs(0, 0, H, C)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        cache.prefill(0, [0], [0, C], qc, kc, vc, out, lse)
    torch.cuda.synchronize()
    peaks, src = load_peaks()
    props = torch.cuda.get_device_properties(0)
    u = str(getattr(props, "uuid", ""))
    clocks = ClockSampler(u if u.startswith("GPU-") else ("GPU-" + u if u else None))
    clocks.start()
    time.sleep(0.4)
    ms = []
    for _ in range(args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        cache.prefill(0, [0], [0, C], qc, kc, vc, out, lse)
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    clk = clocks.stop()
    assert cache.status() == 0
    total = sum(ms)
    tf = flop * args.steps / (total / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return {"metric": "chunked prefill over cached history, TFLOP/s over visible pairs",
            "op": "chunk_prefill", "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps, "higher_is_better": True,
            "dtype": "bf16 MMA; history pages " + ("e4m3 (converted to bf16 in shared memory)" if fp8 else "bf16"),
            "data": "synthetic (seeded N(0,1), pages' shapes)",
            "config": {"workload": "mistral7b layer %d policies, %d cached tokens + %d-row chunk" % (layer, H, C),
                       "kv_dtype": "fp8_e4m3" if fp8 else "bf16", "flop_per_call": flop,
                       "l2": "flushed between calls"},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "kernel": "k_prefill", "peak_source": src + " bf16_tflops (burst)"},
            "clocks": clk}


def run_op_pack(args):
    """sp_pack_seq of Llama-3-8B-shaped sequences (32 layers x 8 KV heads x
    32,768 tokens, the decode workload's policies): HBM-bound, every retained
    row read from the pool and written to the packed buffer.  Also reports
    the transfer-byte ratio dense / packed."""
    import torch
    from head_aware_paged_gb300 import Config, Policy, SegPagedCache, sp_pack_seq
    wl = W.WORKLOADS["llama3_8b_decode_32k"]
    B, n = 4, wl.seq_len
    pols = W.policies(wl)
    pages = 0
    for row in pols:
        for p_ in row:
            pages += B * (-(-n // wl.page) + 1 if p_.kind == W.GLOBAL else
                          -(-p_.sink // wl.page) + -(-p_.window // wl.page) + 2)
    cfg = Config(num_layers=wl.layers, num_q_heads=wl.hq, num_kv_heads=wl.hkv, head_dim=wl.d,
                 page_size=wl.page, max_seqs=B, max_seq_len=n, num_pages=pages + 16,
                 max_tokens=n, max_batch=B)
    c = SegPagedCache(cfg)
    cp = [[Policy(p_.kind, p_.sink, p_.window) for p_ in row] for row in pols]
    for b in range(B):
        c.set_policy(b, cp)
        for l in range(wl.layers):
            k = W.normal((n, wl.hkv, wl.d), W.tensor_seed(0, "k", b, l), device="cuda")
            v = W.normal((n, wl.hkv, wl.d), W.tensor_seed(0, "v", b, l), device="cuda")
            c.build(b, l, k, v)
            del k, v
    torch.cuda.synchronize()
    sizes = [sp_pack_seq(c.handle, b, None) for b in range(B)]
    bufs = [c.pack(b) for b in range(B)]            # also the warm-up
    torch.cuda.synchronize()
    hdr = bufs[0][:96].cpu().numpy().view(np.int64)
    payload = int(hdr[9])
    dense = n * wl.layers * wl.hkv * 2 * wl.d * 2
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        for b in range(B):
            sp_pack_seq(c.handle, b, bufs[b])
    torch.cuda.synchronize()
    peaks, src = load_peaks()
    ms = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for b in range(B):
            sp_pack_seq(c.handle, b, bufs[b])
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    assert c.status() == 0
    total = sum(ms)
    moved = 2 * payload * B             # read from the pool + write to the buffer
    gbs = moved * args.steps / (total / 1e3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"metric": "Pack of trimmed per-head pages for transfer, GB/s moved (read + write)",
            "op": "pack", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1), pages' shapes)",
            "config": {"workload": "llama3_8b_decode_32k policies, %d sequences x 32 layers x %d tokens" % (B, n),
                       "packed_bytes_per_seq": sizes[0], "payload_bytes_per_seq": payload,
                       "dense_kv_bytes_per_seq": dense, "transfer_ratio_dense_over_packed": dense / payload,
                       "l2": "flushed between steps"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": None, "kernel": "k_transfer",
                         "peak_source": "%s hbm_gbs" % src}}


def run_op_select(args):
    """sp_select_heavy_hitters on one 32,768-token prompt (Hq 32 / Hkv 8,
    d 128), observation window 64 rows, top-2048 (the retrieval heads of the
    ragged mixed workload).  Work: two QK^T passes over every visible
    (observation row, key) pair, 2 * 2d FLOP each."""
    import torch
    from head_aware_paged_gb300 import sp_select_heavy_hitters
    n, n_obs, hq, hkv, d, topk = 32768, 64, 32, 8, 128, 2048
    q = W.normal((n_obs, hq, d), 1, device="cuda")
    k = W.normal((n, hkv, d), 2, scale=0.5, device="cuda")
    flop = 2 * 2 * 2 * d * hq * sum(n - n_obs + oi + 1 for oi in range(n_obs))
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        sp_select_heavy_hitters(q, k, topk, 0)
    torch.cuda.synchronize()
    peaks, src = load_peaks()
    ms = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        sp_select_heavy_hitters(q, k, topk, 0)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    total = sum(ms)
    tf = flop * args.steps / (total / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return {"metric": "Heavy-hitter retrieval selection, TFLOP/s over visible (row, key) pairs",
            "op": "select", "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1), K x 0.5)",
            "config": {"workload": "one prompt n=%d, n_obs=%d, Hq %d / Hkv %d, d %d, top-%d" % (n, n_obs, hq, hkv, d, topk),
                       "flop_per_call": flop, "l2": "flushed between calls"},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "traffic": None, "kernel": "k_hh_tile (mma.sync)",
                         "peak_source": "%s bf16_tflops" % src}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 5 for the 64-layer 128K prefill, 64 for the decode "
                         "workload -- its configuration's step count -- else 20)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama33_70b_prefill_128k",
                    choices=["llama33_70b_prefill_128k", "mistral7b_prefill_8k", "llama3_8b_decode_32k"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="leave out the end-to-end leg (short runs and profiling cases)")
    ap.add_argument("--no-decode-record", action="store_true",
                    help="multi-layer prefill workload: leave out the decode record")
    ap.add_argument("--layers", default="",
                    help="prefill workload: run the first N layers (\"N\") or layers a..b-1 (\"a:b\") "
                         "instead of all (short runs and small profiling cases)")
    ap.add_argument("--decode-layers", type=int, default=0,
                    help="decode workload: run only the first N layers (profiling a small case)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="decode workload: page element type (fp8 = e4m3 codes with per-channel scales)")
    ap.add_argument("--op", default="", choices=["", "rope_realign", "pack", "select", "chunk_prefill"],
                    help="time one library operation instead of the attention step")
    args = ap.parse_args()
    if args.steps is None:
        if args.op or args.impl == "reference":
            args.steps = 20 if args.workload != "llama33_70b_prefill_128k" or args.op else 5
        elif args.workload == "llama3_8b_decode_32k":
            args.steps = 64
        elif args.workload == "llama33_70b_prefill_128k":
            args.steps = 5
        else:
            args.steps = 20
    if args.warmup < 3:
        args.warmup = 3
    if args.op:
        line = {"rope_realign": run_op_rope, "pack": run_op_pack, "select": run_op_select,
                "chunk_prefill": run_op_chunk}[args.op](args)
        print(json.dumps(line), flush=True)
        return
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, ws, rank)
    else:
        ws, rank, _ = dist_setup()
        line = run_ours(args, ws, rank)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)
    if args.impl != "reference" and ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
