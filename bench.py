"""Benchmark of the head-aware paged attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mistral7b_prefill_8k|llama3_8b_decode_32k|llama33_70b_prefill_128k]

Prints ONE JSON line (rank 0).  Default workload: the Mistral-7B-shaped
prefill layer (Hq 32 / Hkv 8, d 128, one sequence of 8192 tokens, page 64,
1 GLOBAL + 7 LOCAL(4, 1024) KV heads).  One step is one pass of the whole
path over that batch: causal prefill of the 8192-token chunk, the trimmed
KV write of the chunk (page allocation + scatter), one decode token
(append + split-KV decode), and the release of the sequence's pages.  The
head-class policy is set once, offline, before timing.

Metric: visible-pair TFLOP/s (FLOP = 4 d per visible (query, key) pair, for
the prefill rows and the decode row) for prefill workloads; visible-KV GB/s
(2 d bytes of K and V per visible key and head) for the decode workload.
Timing: CUDA events on the launching stream after W warm-up steps; L2 is
flushed (256 MB write) between steps, outside the timed events.  With
--gpus N > 1 (torchrun), every rank runs the same workload on its own GPU
(replicas; the path has no cross-GPU exchange) and the value is the sum of
the ranks' work over the slowest rank's time.

--impl reference times the CPU oracle (plain fp32 C, all host cores) on a
bounded sample of the same workload, in the same units.
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

class PrefillStep:
    """Prefill + trimmed KV write + one decode token + release, one sequence."""

    def __init__(self, wl, layer_policies, device="cuda"):
        import torch
        from head_aware_paged_gb300 import Config, Policy, SegPagedCache
        self.wl = wl
        L = wl.seq_len
        self.L = L
        pol = [[Policy(p.kind, p.sink, p.window, None if p.idx is None else p.idx.tolist())
                for p in layer_policies]]
        pages = 0
        for p in layer_policies:
            pages += (L + 1 + wl.page - 1) // wl.page + 2
        self.cfg = Config(num_layers=1, num_q_heads=wl.hq, num_kv_heads=wl.hkv, head_dim=wl.d,
                          page_size=wl.page, max_seqs=2, max_seq_len=L + 64, num_pages=2 * pages,
                          max_idx_per_seq=max(1, sum(0 if p.idx is None else len(p.idx)
                                                     for p in layer_policies)),
                          max_tokens=L, max_batch=1)
        self.cache = SegPagedCache(self.cfg)
        self.cache.set_policy(0, pol)
        self.cache.set_policy(1, pol)            # the second request slot of the e2e leg
        self.q, self.k, self.v = W.qkv(wl, L + 1, 0, 0, device=device)
        self.q1 = self.q[L:].contiguous()
        self.k1 = self.k[L:].contiguous()
        self.v1 = self.v[L:].contiguous()
        self.q, self.k, self.v = (self.q[:L].contiguous(), self.k[:L].contiguous(),
                                  self.v[:L].contiguous())
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(L, wl.hq, dtype=torch.float32, device=device)
        self.out1 = torch.empty_like(self.q1)
        self.lse1 = torch.empty(1, wl.hq, dtype=torch.float32, device=device)
        pairs = self.cache.count_prefill_pairs(0, 0, 0, L)
        dec_pairs = self.cache.count_decode_bytes(0, [0], [L]) // (2 * wl.d * 2) * (wl.hq // wl.hkv)
        self.prefill_flop = 4 * wl.d * pairs
        self.work = 4 * wl.d * (pairs + dec_pairs)      # FLOP per step
        self.kernels_per_step = 7                        # prefill, 2x(alloc+scatter), decode, release
        self.unit = "TFLOP/s"

    def run(self, ev_pf=None):
        c = self.cache
        if ev_pf is not None:
            ev_pf[0].record()
        c.prefill(0, [0], [0, self.L], self.q, self.k, self.v, self.out, self.lse)
        if ev_pf is not None:
            ev_pf[1].record()
        c.append_kv(0, [0], [0, self.L], self.k, self.v)
        c.append_kv(0, [0], [0, 1], self.k1, self.v1)
        c.decode(0, [0], self.q1, self.out1, self.lse1)
        c.release(0)

    # host-buffer (end-to-end) variant: every step uploads its q/k/v from
    # pinned host memory and reads out/lse back; consecutive steps run as two
    # requests in flight (sequence slots 0 and 1, two device buffer sets), so
    # step i+1's upload and step i-1's download overlap step i's kernels
    def setup_e2e(self):
        import torch
        pin = lambda t: t.cpu().pin_memory()
        self.h_in = [pin(t) for t in (self.q, self.k, self.v, self.q1, self.k1, self.v1)]
        self.dev = [[torch.empty_like(t) for t in (self.q, self.k, self.v, self.q1, self.k1, self.v1,
                                                    self.out, self.lse, self.out1, self.lse1)]
                    for _ in range(2)]
        self.h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory()
                       for t in (self.out, self.lse, self.out1, self.lse1)] for _ in range(2)]
        self.streams = [torch.cuda.Stream() for _ in range(3)]        # upload, kernels, download
        self.ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.h_out[0])

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
        for i in range(n):
            b = i % 2
            q, k, v, q1, k1, v1, out, lse, out1, lse1 = self.dev[b]
            with torch.cuda.stream(sh):
                if i >= 2:
                    sh.wait_event(self.ev["done"][b])      # step i-2 has read these inputs
                for d, h in zip((q, k, v, q1, k1, v1), self.h_in):
                    d.copy_(h, non_blocking=True)
                self.ev["in"][b].record(sh)
            sc.wait_event(self.ev["in"][b])
            if i >= 2:
                sc.wait_event(self.ev["out"][b])           # step i-2's outputs are home
            c.prefill(0, [b], [0, self.L], q, k, v, out, lse, stream=sc)
            c.append_kv(0, [b], [0, self.L], k, v, stream=sc)
            c.append_kv(0, [b], [0, 1], k1, v1, stream=sc)
            c.decode(0, [b], q1, out1, lse1, stream=sc)
            c.release(b, stream=sc)
            self.ev["done"][b].record(sc)
            sd.wait_event(self.ev["done"][b])
            with torch.cuda.stream(sd):
                for h, d in zip(self.h_out[b], (out, lse, out1, lse1)):
                    h.copy_(d, non_blocking=True)
                self.ev["out"][b].record(sd)
        for st_ in self.streams:
            cur.wait_stream(st_)
        end.record(cur)
        return start, end

    # CPU oracle sample of the same workload: rows spread over the sequence
    def oracle_sample(self, layer_policies, target_s: float, threads: int):
        import oracle
        from oracle import accounting
        pt = [(p.kind, p.sink, p.window, None if p.idx is None else p.idx.tolist())
              for p in layer_policies]
        qf = self.q.float().cpu().numpy()
        kf = self.k.float().cpu().numpy()
        vf = self.v.float().cpu().numpy()
        L = self.L
        rng = np.random.default_rng(5)

        def run_rows(nrows):
            rows = np.sort(rng.choice(L, size=nrows, replace=False))
            t0 = time.perf_counter()
            oracle.attend(qf[rows], kf, vf, rows, pt, "f32", threads=threads)
            dt = time.perf_counter() - t0
            pairs = 0
            grp = self.wl.hq // self.wl.hkv
            for p in pt:
                pairs += grp * int(accounting.vis_count_closed(p[0], p[1], p[2], p[3], rows).sum())
            return dt, 4 * self.wl.d * pairs, nrows

        dt, fl, n = run_rows(16)
        n2 = int(min(L, max(16, 16 * target_s / max(dt, 1e-3))))
        return run_rows(n2), qf, kf, vf, pt


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
        c = self.cache
        for l in range(self.layers):
            c.append_kv(l, self.seqs, self.cu, self.kn, self.vn)
            if ev_pf is not None and l == 0:
                ev_pf[0].record()
            c.decode(l, self.seqs, self.qs, self.out, self.lse)
            if ev_pf is not None and l == 0:
                ev_pf[1].record()
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
    """The prefill step runs one layer: the first whose policy has a GLOBAL KV
    head (every layer has the same shapes; this one carries the full-causal
    work), else layer 0."""
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


# ---------------------------------------------------------------- main arms

def run_ours(args, ws, rank):
    import torch
    from head_aware_paged_gb300 import build as _b
    if rank == 0:
        _b.build()
    barrier(ws)
    torch.cuda.init()
    wl = W.WORKLOADS[args.workload]
    decode = wl.decode_steps > 0 and wl.name.startswith("llama3_8b")
    if args.kv_dtype == "fp8" and not decode:
        raise SystemExit("--kv-dtype fp8 applies to the decode workload and --op chunk_prefill "
                         "(the prefill step has no cached history)")
    if decode:
        st = DecodeStep(wl, layers=args.decode_layers or None, fp8=args.kv_dtype == "fp8")
    else:
        layer = bench_layer(wl)
        st = PrefillStep(wl, W.policies(wl)[layer])
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    assert st.cache.status() == 0

    n_steps = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_steps)]
    evk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_steps)]
    work = []
    kern_work = []
    props = torch.cuda.get_device_properties(0)
    uuid = None
    try:
        u = str(props.uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    clocks = ClockSampler(uuid if rank == 0 else None)
    if rank == 0:
        clocks.start()
        time.sleep(0.4)
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(n_steps):
        flush.random_(0, 255) if i == 0 else flush.fill_(i & 0xFF)
        if decode:
            work.append(st.step_bytes(st.t))
            kern_work.append(st.cache.count_decode_bytes(0, st.seqs, [st.t] * st.B))
        else:
            work.append(st.work)
            kern_work.append(st.prefill_flop)
        ev[i][0].record(stream)
        st.run(evk[i])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if rank == 0 else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in evk]
    total_ms = reduce_max(float(sum(step_ms)), ws)
    assert st.cache.status() == 0
    scale = 1e-12 if not decode else 1e-9
    value = job_rate(float(sum(work)), float(sum(step_ms)), ws) * scale

    # end-to-end through the same C-ABI calls with host buffers (prefill only)
    e2e = None
    if not decode:
        st.setup_e2e()
        st.run_e2e_steps(2)
        torch.cuda.synchronize()
        e2e_steps = max(3, min(n_steps, 10))
        barrier(ws)
        e0, e1 = st.run_e2e_steps(e2e_steps)
        torch.cuda.synchronize()
        assert st.cache.status() == 0
        e2e = {"value": job_rate(float(st.work * e2e_steps), e0.elapsed_time(e1), ws) * scale,
               "unit": st.unit,
               "h2d_bytes_per_step": st.h2d_bytes, "d2h_bytes_per_step": st.d2h_bytes}
    else:
        st.setup_e2e()
        st.run_e2e_steps(1)
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1, w = st.run_e2e_steps(3)
        torch.cuda.synchronize()
        assert st.cache.status() == 0
        e2e_rate = job_rate(float(w), e0.elapsed_time(e1), ws)
        bytes_in, bytes_out = st.h2d_bytes, st.d2h_bytes
        e2e = {"value": e2e_rate * scale, "unit": st.unit,
               "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out}

    if rank != 0:
        return None
    peaks, src = load_peaks()
    kern_avg_ms = float(np.mean(kern_ms))
    if decode:
        achieved = float(np.mean(kern_work)) / (kern_avg_ms / 1e3) / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": load_traffic("k_decode", wl.name + ("_fp8" if st.fp8 else "")),
                "kernel": "k_decode", "peak_source": src + " hbm_gbs",
                "algorithmic_bytes_per_launch": int(np.mean(kern_work)),
                "avg_launch_ms": kern_avg_ms}
    else:
        achieved = st.prefill_flop / (kern_avg_ms / 1e3) / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": load_traffic("k_prefill", wl.name),
                "kernel": "k_prefill", "peak_source": src + " bf16_tflops (burst)",
                "algorithmic_flop_per_launch": st.prefill_flop, "avg_launch_ms": kern_avg_ms}

    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(st, wl, decode)
    line = {
        "metric": "SegPaged prefill TFLOP/s & decode visible-KV GB/s, % of GB300 roofline",
        "value": value, "unit": st.unit, "n_gpus": ws, "steps": n_steps, "warmup": args.warmup,
        "ms_per_step": total_ms / n_steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 K/V pages, f16 MMA" if decode and st.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), pages' shapes)",
        "config": config_dict(wl, decode, st),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": st.kernels_per_step * n_steps, "clocks": clk,
    }
    return line


def config_dict(wl, decode, st):
    d = {"workload": wl.name, "hq": wl.hq, "hkv": wl.hkv, "head_dim": wl.d, "page_size": wl.page,
         "l2": "flushed between steps (256 MB write outside the timed events)",
         "parallelism": "replicas (no cross-GPU exchange on this path)"}
    if decode:
        d.update({"layers": st.layers, "batch": wl.seqs, "cached_tokens": wl.seq_len,
                  "global_units": wl.n_global, "local": [wl.local_sink, wl.local_window],
                  "step": "all layers: append 1 token/seq + split-KV decode",
                  "kv_dtype": "fp8_e4m3" if st.fp8 else "bf16"})
        if st.fp8:
            d["workload"] = wl.name + "_fp8"
            d["kv_scales"] = "%.6g for every channel of K and V" % FP8_SCALE
    else:
        layer = bench_layer(wl)
        d.update({"seq_len": wl.seq_len, "layer": layer, "global_kv_heads_in_layer": sum(
            1 for p in W.policies(wl)[layer] if p.kind == W.GLOBAL),
                  "local": [wl.local_sink, wl.local_window],
                  "step": "prefill + trimmed KV write + 1 decode token + release"})
    return d


def cpu_baseline(st, wl, decode, target_s=12.0):
    threads = os.cpu_count() or 1
    if decode:
        import oracle
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
    (dt, fl, n), *_ = st.oracle_sample(W.policies(wl)[0], target_s, threads)
    (dt1, fl1, n1), *_ = st.oracle_sample(W.policies(wl)[0], target_s / threads, 1)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d query rows (all %d heads), fp32 C oracle" % (n, st.L, wl.hq),
            "one_thread": {"value": fl1 / dt1 / 1e12, "cores": 1,
                           "sample": "%d of %d query rows (all %d heads)" % (n1, st.L, wl.hq)}}


def run_reference(args, ws, rank):
    """The CPU oracle as the reference arm: each step one bounded sample."""
    if ws > 1 and rank != 0:
        return None
    import oracle
    from oracle import accounting
    wl = W.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    decode = wl.name.startswith("llama3_8b")
    rng = np.random.default_rng(1)
    if decode:
        L = wl.seq_len
        pol = W.policies(wl)[0]
        pt = [(p.kind, p.sink, p.window, None) for p in pol]
        k = W.normal((L, wl.hkv, wl.d), W.tensor_seed(0, "k", 0, 0)).float().numpy()
        v = W.normal((L, wl.hkv, wl.d), W.tensor_seed(0, "v", 0, 0)).float().numpy()
        q = W.normal((1, wl.hq, wl.d), 11).float().numpy()
        nb = sum(int(accounting.vis_count_closed(p[0], p[1], p[2], p[3], np.array([L - 1]))[0])
                 for p in pt) * 2 * wl.d * 2

        def one():
            oracle.attend(q, k, v, [L - 1], pt, "f32", threads=threads)
            return nb
        unit, scale, sample = "GB/s", 1e-9, "one decode query of one sequence, layer 0, fp32 C oracle"
    else:
        L = wl.seq_len
        pt = [(p.kind, p.sink, p.window, None) for p in W.policies(wl)[bench_layer(wl)]]
        q, k, v = (t.float().numpy() for t in W.qkv(wl, L, 0, 0))
        grp = wl.hq // wl.hkv
        nrows = 48

        def one():
            rows = np.sort(rng.choice(L, size=nrows, replace=False))
            oracle.attend(q[rows], k, v, rows, pt, "f32", threads=threads)
            return 4 * wl.d * sum(grp * int(accounting.vis_count_closed(p[0], p[1], p[2], p[3], rows).sum())
                                  for p in pt)
        unit, scale, sample = "TFLOP/s", 1e-12, "48 random query rows (all heads) per step, fp32 C oracle"
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    work = 0
    for _ in range(args.steps):
        work += one()
    dt = time.perf_counter() - t0
    value = work * scale / dt
    return {"impl": "reference", "metric": "SegPaged prefill TFLOP/s & decode visible-KV GB/s, % of GB300 roofline",
            "value": value, "unit": unit, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0,1), pages' shapes)",
            "config": {"workload": wl.name, "hq": wl.hq, "hkv": wl.hkv, "head_dim": wl.d},
            "cpu_baseline": {"value": value, "unit": unit, "kind": "oracle", "cores": threads,
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


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
                    help="timed steps (default 20; the decode workload 64, the step count of "
                         "its configuration)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mistral7b_prefill_8k",
                    choices=["mistral7b_prefill_8k", "llama3_8b_decode_32k", "llama33_70b_prefill_128k"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-layers", type=int, default=0,
                    help="decode workload: run only the first N layers (profiling a small case)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="decode workload: page element type (fp8 = e4m3 codes with per-channel scales)")
    ap.add_argument("--op", default="", choices=["", "rope_realign", "pack", "select", "chunk_prefill"],
                    help="time one library operation instead of the attention step")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 64 if (args.workload == "llama3_8b_decode_32k" and not args.op
                            and args.impl == "ours") else 20
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
