#!/usr/bin/env python
"""Benchmark of the self-speculative decoding hot path on GB300.

One step = one pass of the whole hot path over one batch of the synthetic
workload (Llama-3.1-8B attention shape, batch 128, context 32768, gamma 4 by
default): SnapKV selection of the draft cache (window scores, max-pool, top-K,
gather), gamma draft steps (draft attention over the compacted cache + draft
token draw), verify attention over the full cache (gamma+1 rows), and
rejection sampling.  The headline metric is verified tokens per second per
layer (B * (gamma+1) per step); per-kernel KV-read GB/s and the HBM roofline
fraction of the verify kernel are reported beside it.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

With --gpus N > 1 every rank runs one full batch on its own GPU (weak scaling,
no collective on the data path: the sequences of a batch are independent); the
timed region is bracketed by barriers and the max over ranks is reported.
Started without WORLD_SIZE in the environment, `--gpus N` re-launches itself
under torch.distributed.run with N processes; under a launcher, WORLD_SIZE must
equal N.  --impl reference times the float64 CPU oracle on a bounded sample of
the same workload (rank 0 only), spread over the host cores by a process pool.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "verified tokens/s/layer and KV-read GB/s (% of GB300 HBM peak) at batch x ctx"
UNIT = "tokens/s/layer"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth; the measured copy figure is the roofline denominator
FALLBACK_BF16_SUSTAINED_TFLOPS = 1700.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="b128_ctx32k",
                   choices=["b32_ctx8k", "b128_ctx32k", "ragged_b256_ctx4k_64k", "round_b32_ctx16k_32layers"],
                   help="b128_ctx32k: batch 128 x 32k (default); round_b32_ctx16k_32layers: full 32-layer "
                        "speculation round")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-round", action="store_true",
                   help="skip the 32-layer round block that the default line carries beside its main workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample", type=int, default=8, help="sequences in the oracle sample")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def launch_ranks(n, argv, script=None):
    """Run `script` (this file by default) with `argv` as n ranks on this node under
    torch.distributed.run; rank 0 prints the line.  Returns the launcher's exit code."""
    script = os.path.abspath(__file__) if script is None else script
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), script] + list(argv)
    return subprocess.call(cmd)


def check_world(args, world):
    if world != args.gpus:
        raise SystemExit("bench.py: --gpus %d but WORLD_SIZE=%d: launch one rank per GPU" % (args.gpus, world))


def run_timed(step, steps, world, device, timer, sync):
    """The timed region of both GPU arms: a barrier and a device sync on both sides of exactly
    `steps` calls of step(i), timed by `timer` (start(), stop(), elapsed_ms()) on the launching
    stream; returns the max over ranks of the per-step time in ms."""
    barrier(world)
    sync()
    timer.start()
    for i in range(steps):
        step(i)
    timer.stop()
    sync()
    barrier(world)
    return max_over_ranks(timer.elapsed_ms(), world, device) / steps


class CudaTimer:
    """CUDA events recorded on the current stream (the stream the library calls launch on)."""

    def __init__(self):
        self.s = torch.cuda.Event(enable_timing=True)
        self.e = torch.cuda.Event(enable_timing=True)

    def start(self):
        self.s.record()

    def stop(self):
        self.e.record()

    def elapsed_ms(self):
        self.e.synchronize()
        return self.s.elapsed_time(self.e)


# ------------------------------------------------------------------ peaks and clocks
def bf16_peak():
    """Sustained bf16 tensor throughput (TFLOP/s) from MEASURED_PEAKS.json, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return FALLBACK_BF16_SUSTAINED_TFLOPS


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "mgd_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ the GPU workload
class Workload:
    def __init__(self, name, device, seed=0):
        from long_context_speculative_split_gb300 import mgd, ops
        from long_context_speculative_split_gb300 import workloads as wl
        self.ops, self.mgd, self.wl = ops, mgd, wl
        c = self.cfg = wl.WORKLOADS[name]
        self.dev = device
        self.B, self.Hq, self.Hkv, self.D = c["B"], c["Hq"], c["Hkv"], c["D"]
        self.gamma, self.K, self.W, self.P, self.V = c["gamma"], c["K"], c["W"], c["pool"], c["V"]
        self.T = self.gamma + 1
        self.kv_len = wl.lengths(c, seed)
        self.cap = wl.capacity(c, seed)
        self.kv_len_d = self.kv_len.to(device)
        self.k, self.v = wl.kv_cache(c, device, seed, kv_len=self.kv_len, cap=self.cap)
        self.q = wl.queries(c, device, seed)
        self.qw = wl.window_queries(c, device, seed)
        self.qd = torch.stack([wl.draft_queries(c, device, seed, step=s)[:, 0] for s in range(self.gamma)])
        self.t, self.d = wl.logits(c, device, seed)
        self.u = wl.uniforms(c, device, seed)
        B, Hq, Hkv, D, K = self.B, self.Hq, self.Hkv, self.D, self.K
        f32, i32 = torch.float32, torch.int32
        self.sel = dict(sel_idx=torch.empty((B, Hkv, K), dtype=i32, device=device),
                        k_draft=torch.zeros((B, Hkv, K, D), dtype=self.k.dtype, device=device),
                        v_draft=torch.zeros((B, Hkv, K, D), dtype=self.k.dtype, device=device),
                        draft_len=torch.empty((B,), dtype=i32, device=device), scores=None)
        self.dout = torch.empty((B, Hq, D), dtype=f32, device=device)
        self.dlse = torch.empty((B, Hq), dtype=f32, device=device)
        self.vout = torch.empty((B, self.T, Hq, D), dtype=f32, device=device)
        self.vlse = torch.empty((B, self.T, Hq), dtype=f32, device=device)
        self.tok = torch.empty((B, self.gamma), dtype=i32, device=device)
        self.out_tok = torch.empty((B, self.T), dtype=i32, device=device)
        self.nacc = torch.empty((B,), dtype=i32, device=device)
        ws = ops.workspace
        self.ws_snap = ws(mgd.mgd_snapkv_workspace_size(B, Hq, Hkv, D, self.cap, self.W), device)
        self.ws_draft = ws(mgd.mgd_draft_workspace_size(B, Hq, Hkv, D, K), device)
        self.ws_verify = ws(mgd.mgd_verify_workspace_size(B, self.T, Hq, Hkv, D, self.cap), device)
        self.ws_spec = ws(mgd.mgd_spec_workspace_size(B, self.gamma, self.V), device)
        L = self.kv_len.double()
        esz = self.k.element_size()
        self.bytes_verify = float((2 * Hkv * L * D * esz).sum())
        Keff = torch.clamp(L, max=K)
        self.bytes_draft = float((2 * Hkv * Keff * D * esz).sum())
        # K read once (both scoring passes of a slice share one HBM read) + the gather (K and V rows read and written)
        self.bytes_snap = float((Hkv * L * D * esz).sum() + 4 * Hkv * Keff.sum() * D * esz)
        # window scores: two contractions of W*G rows x D per key (pass 1 over all L keys, pass 2 over L - W)
        self.flops_snap = float((2 * self.W * (Hq // Hkv) * D * Hkv * (2 * L - self.W)).sum())
        # rejection sample: the gamma + 1 target rows (the draft rows' normalisers come from the draws)
        self.bytes_spec = float(B * (self.gamma + 1) * self.V * 4)
        # SnapKV (one-read scorer + select), gamma x (draft attention + one-row draw), verify,
        # rejection sample (statistics and finish)
        self.launches_per_step = 2 + self.gamma * 1 + self.gamma * 1 + 1 + 2

    def step(self, ev=None):
        ops = self.ops
        if ev:
            ev[0].record()
        ops.snapkv_select(self.qw, self.k, self.v, self.kv_len_d, self.W, self.P, self.K, ws=self.ws_snap,
                          out=self.sel)
        if ev:
            ev[1].record()
        for s in range(self.gamma):
            ops.draft_attn(self.qd[s], self.sel["k_draft"], self.sel["v_draft"], self.sel["draft_len"],
                           ws=self.ws_draft, out=self.dout, lse=self.dlse)
            ops.draft_draw(self.d, self.u, draft_tokens=self.tok, row=s, ws=self.ws_spec)
        if ev:
            ev[2].record()
        ops.verify_attn(self.q, self.k, self.v, self.kv_len_d, ws=self.ws_verify, out=self.vout, lse=self.vlse)
        if ev:
            ev[3].record()
        ops.rejection_sample(self.t, self.d, self.tok, self.u, ws=self.ws_spec, out_tokens=self.out_tok,
                             num_accepted=self.nacc, reuse_draft_stats=True)
        if ev:
            ev[4].record()

    def _per_launch_ms(self, fn, reps, flush_l2=False):
        """Average device time of `reps` back-to-back calls between two events on the launching
        stream (median of 3 trials).  A short GPU sleep ahead of the first event keeps the stream
        busy while the host queues every call (a call costs tens of microseconds of host time,
        more than a small kernel runs), so the events bracket device work only: each launch,
        its workspace reset and the gaps between them.  With `flush_l2` a 512 MB write evicts
        L2 first."""
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(2):
            fn()
        flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=self.dev) if flush_l2 else None
        sleep_cycles = int(2.1e9 * (2e-3 + reps * 60e-6))  # covers the host's queueing of `reps` calls
        times = []
        for _ in range(3):
            if flush is not None:
                flush.fill_(1.0)
            torch.cuda._sleep(sleep_cycles)
            s.record()
            for _ in range(reps):
                fn()
            e.record()
            e.synchronize()
            times.append(s.elapsed_time(e) / reps)
        return statistics.median(times)

    def time_decode(self, reps=3):
        """Plain decode attention (one query row) over the full cache: T_T of the speedup model."""
        ops = self.ops
        q1 = self.q[:, :1].contiguous()
        out = torch.empty((self.B, 1, self.Hq, self.D), dtype=torch.float32, device=self.dev)
        lse = torch.empty((self.B, 1, self.Hq), dtype=torch.float32, device=self.dev)
        ws = ops.workspace(self.mgd.mgd_verify_workspace_size(self.B, 1, self.Hq, self.Hkv, self.D, self.cap),
                           self.dev)
        return self._per_launch_ms(lambda: ops.verify_attn(q1, self.k, self.v, self.kv_len_d, ws=ws, out=out,
                                                           lse=lse), reps)

    def time_streaming(self, reps=10):
        """StreamingLLM-style draft-cache build (4 sinks + recent rows, same budget K)."""
        ops = self.ops
        out = dict(sel_idx=torch.empty_like(self.sel["sel_idx"]), k_draft=torch.empty_like(self.sel["k_draft"]),
                   v_draft=torch.empty_like(self.sel["v_draft"]), draft_len=torch.empty_like(self.sel["draft_len"]))
        return self._per_launch_ms(lambda: ops.streaming_select(self.k, self.v, self.kv_len_d, 4, self.K, out=out),
                                   reps, flush_l2=True)

    def time_topk_draft(self, reps=3):
        """One dynamic top-K draft step (NEXT-4): select the K rows the draft query attends to most over
        the full cache, then attend over them; compared with the static draft step and plain decode."""
        ops = self.ops
        q = self.qd[0]
        out = dict(out=torch.empty_like(self.dout), lse=torch.empty_like(self.dlse),
                   sel_idx=torch.empty_like(self.sel["sel_idx"]), k_draft=torch.empty_like(self.sel["k_draft"]),
                   v_draft=torch.empty_like(self.sel["v_draft"]), draft_len=torch.empty_like(self.sel["draft_len"]))
        ws = ops.workspace(self.mgd.mgd_topk_draft_workspace_size(self.B, self.Hq, self.Hkv, self.D, self.cap,
                                                                  self.K), self.dev)
        return self._per_launch_ms(lambda: ops.topk_draft_attn(q, self.k, self.v, self.kv_len_d, self.K, ws=ws,
                                                                out=out), reps)

    def time_draft_only(self, reps=20):
        """Draft attention alone, for its own roofline figure.  Back-to-back launches cycle
        through copies of the draft cache totalling at least 256 MB (twice L2), so every
        launch streams its K/V from HBM."""
        ops = self.ops
        kd, vd = self.sel["k_draft"], self.sel["v_draft"]
        ncopy = max(1, -(-256 * 2 ** 20 // int(2 * kd.numel() * kd.element_size())))
        caches = [(kd, vd)] + [(kd.clone(), vd.clone()) for _ in range(ncopy - 1)]
        it = [0]

        def one():
            k, v = caches[it[0] % len(caches)]
            it[0] += 1
            ops.draft_attn(self.qd[0], k, v, self.sel["draft_len"], ws=self.ws_draft, out=self.dout, lse=self.dlse)

        ms = self._per_launch_ms(one, reps, flush_l2=True)
        del caches
        return ms


def run_e2e(w, steps, warmup):
    """Same metric through the public API with pinned host inputs copied in every step."""
    host = {}
    for name in ("k", "v", "q", "qw", "qd", "t", "d", "u"):
        src = getattr(w, name)
        h = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
        h.copy_(src)
        host[name] = h
    host["kv_len"] = w.kv_len.clone().pin_memory()
    out_tok_h = torch.empty(w.out_tok.shape, dtype=torch.int32, pin_memory=True)
    nacc_h = torch.empty(w.nacc.shape, dtype=torch.int32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_tok_h.numel() * 4 + nacc_h.numel() * 4

    def one():
        for name in ("k", "v", "q", "qw", "qd", "t", "d", "u"):
            getattr(w, name).copy_(host[name], non_blocking=True)
        w.kv_len_d.copy_(host["kv_len"], non_blocking=True)
        w.step()
        out_tok_h.copy_(w.out_tok, non_blocking=True)
        nacc_h.copy_(w.nacc, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        one()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    del host
    return ms, h2d, d2h


# ------------------------------------------------------------------ the oracle on host cores
def oracle_inputs(cfg, n_seq, seed=0):
    """CPU inputs of the first n_seq sequences of the workload, in shared memory (not timed)."""
    import math

    from long_context_speculative_split_gb300 import workloads as wl
    c = dict(cfg)
    lens = wl.lengths(cfg, seed)[:n_seq]
    c["B"] = n_seq
    c["lens"] = [int(x) for x in lens]
    cap = int(lens.max())
    k, v = wl.kv_cache(c, "cpu", seed, kv_len=lens, cap=cap)
    t, d = wl.logits(c, "cpu", seed)
    inp = dict(k=k, v=v, q=wl.queries(c, "cpu", seed), qw=wl.window_queries(c, "cpu", seed),
               qd=torch.stack([wl.draft_queries(c, "cpu", seed, step=s) for s in range(c["gamma"])]),
               t=t, d=d, u=wl.uniforms(c, "cpu", seed), lens=lens)
    for x in inp.values():
        x.share_memory_()
    inp.update(W=c["W"], pool=c["pool"], K=c["K"], gamma=c["gamma"], G=c["Hq"] // c["Hkv"], Hkv=c["Hkv"],
               scale=1.0 / math.sqrt(c["D"]))
    return inp


def oracle_pair_job(job):
    """The attention side of the path for one (sequence, KV head), by the float64 oracle: SnapKV
    selection, gamma draft attentions over the selected rows, verify attention over the cache."""
    from oracle.attention import attention, draft_attention
    from oracle.snapkv import snapkv_select
    x, b, h = job
    hs = slice(h * x["G"], (h + 1) * x["G"])
    L = x["lens"][b:b + 1]
    n = int(L[0])
    k, v = x["k"][b:b + 1, h:h + 1, :n], x["v"][b:b + 1, h:h + 1, :n]
    sel = snapkv_select(x["qw"][b:b + 1, :, hs], k, v, L, x["W"], x["pool"], x["K"], x["scale"])
    for s in range(x["gamma"]):
        draft_attention(x["qd"][s, b:b + 1, :, hs], sel["k_draft"], sel["v_draft"], sel["draft_len"], x["scale"])
    attention(x["q"][b:b + 1, :, hs], k, v, L, x["scale"])
    return b, h


def oracle_seq_job(job):
    """The sampling side for one sequence, by the float64 oracle: gamma draft draws, then
    rejection sampling of the round."""
    import numpy as np

    from oracle.sampling import draft_draw, rejection_sample
    x, b = job
    d, u = x["d"][b:b + 1], x["u"][b:b + 1]
    toks = [draft_draw(d[:, s:s + 1], u[:, s:s + 1])[0][:, 0] for s in range(x["gamma"])]
    rejection_sample(x["t"][b:b + 1], d, np.stack(toks, axis=1), u)
    return b


def _pool_ready(_):
    import oracle.attention  # noqa: F401  (imports paid before the timed steps)
    import oracle.sampling  # noqa: F401
    import oracle.snapkv  # noqa: F401
    return os.getpid()


class OracleBaseline:
    """The float64 oracle over a sample of n_seq sequences, as it stands, spread over the host
    cores this process may use: one task per (sequence, KV head) for the attention side and one
    per sequence for sampling, in a pool of spawned processes (BLAS one thread each)."""

    def __init__(self, cfg, n_seq, seed=0):
        import torch.multiprocessing as tmp
        self.n_seq, self.cores = n_seq, len(os.sched_getaffinity(0))
        self.inp = oracle_inputs(cfg, n_seq, seed)
        self.pool = tmp.get_context("spawn").Pool(self.cores)
        self.pool.map(_pool_ready, range(self.cores))
        self.pairs = [(self.inp, b, h) for b in range(n_seq) for h in range(self.inp["Hkv"])]
        self.seqs = [(self.inp, b) for b in range(n_seq)]

    def step(self):
        """One pass over the sample; returns wall-clock seconds."""
        t0 = time.perf_counter()
        r1 = self.pool.map_async(oracle_pair_job, self.pairs, chunksize=1)
        r2 = self.pool.map_async(oracle_seq_job, self.seqs, chunksize=1)
        r1.get()
        r2.get()
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()

    def sample_text(self, cfg, sec):
        return ("%d of %d sequences (all %d KV heads, full context), whole path: %d (sequence, KV head) tasks and "
                "%d sampling tasks over %d processes, %.1f s" % (self.n_seq, cfg["B"], cfg["Hkv"], len(self.pairs),
                                                                 len(self.seqs), self.cores, sec))


# ------------------------------------------------------------------ arms
def run_reference(args):
    rank, world, _ = dist_env()
    check_world(args, world)
    if rank != 0:
        return 0
    from long_context_speculative_split_gb300 import workloads as wl
    cfg = wl.WORKLOADS[args.workload]
    T = cfg["gamma"] + 1
    ob = OracleBaseline(cfg, min(args.cpu_sample, cfg["B"]))
    for _ in range(args.warmup):
        ob.step()
    times = [ob.step() for _ in range(args.steps)]
    ob.close()
    sec = sum(times) / len(times)
    value = ob.n_seq * T / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": ob.cores, "kind": "oracle",
                         "sample": ob.sample_text(cfg, sec)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def kv_and_logit_gb(cfg):
    from long_context_speculative_split_gb300 import workloads as wl
    kv = 2 * cfg["Hkv"] * cfg["D"] * 2 * float(wl.lengths(cfg).double().sum())
    logits = cfg["B"] * (2 * cfg["gamma"] + 1) * cfg["V"] * 4
    return kv / 1e9, logits / 1e9


def config_block(cfg):
    lens = cfg["lens"]
    ctx = lens if not isinstance(lens, tuple) else "U[%d, %d]" % lens
    return {"workload": "%s: batch %d, context %s, %dq/%dkv heads, head_dim %d, gamma %d, draft budget K=%d, "
                        "SnapKV window %d, pool %d, vocab %d (Llama-3.1-8B attention shape, synthetic)" % (
                            cfg["name"], cfg["B"], ctx, cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["gamma"], cfg["K"],
                            cfg["W"], cfg["pool"], cfg["V"]),
            "batch": cfg["B"], "ctx": ctx, "gamma": cfg["gamma"], "K": cfg["K"],
            "l2": "inputs larger than L2 (KV %.1f GB, logits %.2f GB); standalone draft timing cycles through "
                  "draft-cache copies of >= 256 MB" % kv_and_logit_gb(cfg),
            "parallelism": "weak: one full batch per GPU"}


def setup_rank(args):
    """This rank's GPU (one per rank, LOCAL_RANK) and, for N > 1, the NCCL process group used
    only for the barriers and the max over ranks around the timed region."""
    rank, world, local = dist_env()
    check_world(args, world)
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU (the oracle arm is --impl reference)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    import __graft_entry__
    __graft_entry__.build()
    return rank, world, local, dev


def run_ours(args):
    rank, world, local, dev = setup_rank(args)
    w = Workload(args.workload, dev, seed=rank)
    for _ in range(args.warmup):
        w.step()
    torch.cuda.synchronize()
    nev = 5
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    ms_step = run_timed(lambda i: w.step(evs[i]), args.steps, world, dev, CudaTimer(), torch.cuda.synchronize)
    clk = clocks.stop()
    phase = [[evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)] for j in range(nev - 1)]
    snap_ms, draft_ms, verify_ms, spec_ms = (statistics.mean(x) for x in phase)
    errs = w.mgd.mgd_workspace_errors(w.ws_verify) | w.mgd.mgd_workspace_errors(w.ws_snap)
    tokens = w.B * w.T
    value = world * tokens / (ms_step / 1e3)
    peak, peak_kind = hbm_peak()
    verify_gbs = w.bytes_verify / (verify_ms / 1e3) / 1e9
    draft_alone_ms = w.time_draft_only()
    draft_gbs = w.bytes_draft / (draft_alone_ms / 1e3) / 1e9
    decode_ms = w.time_decode()
    streaming_ms = w.time_streaming()
    topk_ms = w.time_topk_draft()
    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h = run_e2e(w, max(1, min(args.steps, 5)), 1)
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": world * tokens / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms,
               # host-to-device bytes over the whole step time: the step is bound by this link
               "h2d_gbs_over_step": h2d / (e_ms / 1e3) / 1e9}
    traffic = load_traffic(args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_block(w.cfg),
        "roofline": {"kernel": "verify attention (split-KV, tensor-core mma, TMA)", "bound": "hbm",
                     "achieved": verify_gbs, "peak": peak, "unit": "GB/s", "frac": verify_gbs / peak,
                     "peak_kind": peak_kind + " (sustained read+write copy)",
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": verify_gbs / NOMINAL_HBM_GBS,
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": w.bytes_verify, "ms_per_launch": verify_ms},
        "kernels": {
            "verify_attention": {"ms": verify_ms, "kv_gbs": verify_gbs, "frac_of_peak": verify_gbs / peak,
                                 "frac_of_nominal": verify_gbs / NOMINAL_HBM_GBS,
                                 "verified_tokens_per_s_per_layer": tokens / (verify_ms / 1e3)},
            "draft_attention": {"ms_per_launch_back_to_back": draft_alone_ms, "kv_gbs": draft_gbs,
                                "frac_of_peak": draft_gbs / peak, "frac_of_nominal": draft_gbs / NOMINAL_HBM_GBS,
                                "ms_per_step_all_gamma_incl_draw": draft_ms},
            "snapkv_select": {"ms": snap_ms, "kv_gbs": w.bytes_snap / (snap_ms / 1e3) / 1e9,
                              "score_tflops": w.flops_snap / (snap_ms / 1e3) / 1e12,
                              "score_frac_of_bf16_sustained": w.flops_snap / (snap_ms / 1e3) / 1e12 / bf16_peak()},
            "rejection_sample": {"ms": spec_ms, "gbs": w.bytes_spec / (spec_ms / 1e3) / 1e9},
        },
        "speedup_model": speedup_model(decode_ms, verify_ms, draft_alone_ms, snap_ms, w.gamma),
        "next": {"streaming_select_ms": streaming_ms,
                 "streaming_select_gbs": 2 * w.bytes_draft / (streaming_ms / 1e3) / 1e9,
                 "topk_draft_step_ms": topk_ms,
                 "topk_draft_over_static_draft": topk_ms / draft_alone_ms,
                 "topk_draft_over_decode": topk_ms / decode_ms},
        "gpu_launches": w.launches_per_step * args.steps,
        "device_error_flags": errs,
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_round:  # the 32-layer speculation round (propose, verify, sample, commit), same GPU
        cfg_w, B_w, T_w, Hkv_w = w.cfg, w.B, w.T, w.Hkv
        del w
        torch.cuda.empty_cache()
        line["round"] = round_block(args, dev, world, rank, local)[0]
    else:
        cfg_w, B_w, T_w, Hkv_w = w.cfg, w.B, w.T, w.Hkv
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ob = OracleBaseline(cfg_w, min(args.cpu_sample, B_w))
        ob.step()  # warm-up pass
        sec = ob.step()
        ob.close()
        line["cpu_baseline"] = {"value": ob.n_seq * T_w / sec, "unit": UNIT, "cores": ob.cores, "kind": "oracle",
                                "sample": ob.sample_text(cfg_w, sec)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def round_block(args, dev, world, rank, local):
    """The 32-layer round workload, one full speculation round per step (propose, verify, sample,
    commit), replayed from a CUDA graph that first restores the lengths, so every replay does the
    same work.  Returns (block for the JSON line, ms per round, kernels per round, clocks)."""
    from long_context_speculative_split_gb300 import mgd
    from long_context_speculative_split_gb300 import workloads as wl
    from long_context_speculative_split_gb300.round import SpeculationRound
    cfg = wl.WORKLOADS["round_b32_ctx16k_32layers"]
    r = SpeculationRound(cfg, dev, seed=rank).prepare()
    graph = True
    try:
        r.capture(restore=True)
    except Exception as e:  # eager launches if capture is refused
        graph = "failed: %s" % str(e).splitlines()[0][:120]
        r.graph = None
        torch.cuda.synchronize()

    def one(_i=0):
        if r.graph is None:
            r.restore()
        r.replay()

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ms = run_timed(one, args.steps, world, dev, CudaTimer(), torch.cuda.synchronize)
    clk = clocks.stop()
    nacc = r.nacc.double()
    committed = float((nacc + 1).mean())
    errs = mgd.mgd_workspace_errors(r.ws_commit) | mgd.mgd_workspace_errors(r.ws_verify)
    # the phases of a round timed on their own (proposal; verification and correction; commit)
    phase_ms = [None, None, None]
    if graph is True:
        for i, g in enumerate(r.capture_phases()):
            for _ in range(2):
                g.replay()
            t = CudaTimer()
            torch.cuda.synchronize()
            t.start()
            for _ in range(args.steps):
                g.replay()
            t.stop()
            phase_ms[i] = t.elapsed_ms() / args.steps
    peak, peak_kind = hbm_peak()
    attn_bytes = r.bytes_verify + r.bytes_draft
    block = {
        "workload": "%s: batch %d, context %d, %d layers of %dq/%dkv head_dim %d, gamma %d, draft K=%d, vocab %d, "
                    "draft noise sigma_n=%.4f (mean acceptance 0.9)" % (
                        cfg["name"], r.B, r.cap, r.layers, r.Hq, r.Hkv, r.D, r.gamma, r.K, r.V, cfg["sigma_n"]),
        "cuda_graph": graph,
        "ms_per_round": ms,
        "verified_tokens_per_s_per_layer": world * r.B * r.T / (ms / 1e3) * r.layers,
        "committed_tokens_per_s": world * r.B * committed / (ms / 1e3),
        "mean_tokens_per_round": committed, "omega_expected_at_alpha_0.9": 3.439,
        "ms_per_committed_token": ms / committed,
        "proposal_ms": phase_ms[0], "verify_and_correction_ms": phase_ms[1], "commit_ms": phase_ms[2],
        "attention_kv_gbs": attn_bytes / (ms / 1e3) / 1e9,
        "attention_frac_of_peak": attn_bytes / (ms / 1e3) / 1e9 / peak, "peak_kind": peak_kind,
        "attention_frac_of_nominal": attn_bytes / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        "gpu_launches_per_round": r.launches,
        "device_error_flags": errs,
        "clocks": clk,
    }
    del r
    torch.cuda.empty_cache()
    return block, ms, block["gpu_launches_per_round"], clk


def run_round(args):
    """The 32-layer round workload as the bench line's main measurement."""
    rank, world, local, dev = setup_rank(args)
    block, ms, launches, clk = round_block(args, dev, world, rank, local)
    line = {
        "metric": METRIC, "value": block["verified_tokens_per_s_per_layer"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": block["workload"], "l2": "inputs larger than L2 (68.7 GB KV)",
                   "cuda_graph": block["cuda_graph"], "parallelism": "weak: one full batch per GPU"},
        "round": block,
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def speedup_model(t_decode, t_verify, t_draft, t_select, gamma):
    """MagicDec notes, quick-read summary (Eq. 2 with Eq. 3's draft cost), restricted to attention:
    Speedup = T_T * Omega(gamma, alpha) / (T_select(K) + gamma * T_D(K) + T_V(gamma)), with measured
    attention times and Omega = (1 - alpha^(gamma+1)) / (1 - alpha).  Static selection runs once per
    prefill, so it is shown both charged to every round and amortised away."""
    out = {"T_T_decode_ms": t_decode, "T_V_verify_ms": t_verify, "T_D_draft_ms": t_draft,
           "T_select_ms": t_select, "T_V_over_T_T": t_verify / t_decode, "T_D_over_T_T": t_draft / t_decode,
           "scope": "attention only (no linear layers: no weights in scope)"}
    for alpha in (0.8, 0.9):
        om = (1 - alpha ** (gamma + 1)) / (1 - alpha)
        out["alpha_%.1f" % alpha] = {
            "omega": om,
            "speedup_selection_amortised": t_decode * om / (gamma * t_draft + t_verify),
            "speedup_selection_every_round": t_decode * om / (t_select + gamma * t_draft + t_verify),
            # T_SD per round and per generated token (T_SD / Omega), attention only, selection amortised
            "round_ms": gamma * t_draft + t_verify,
            "ms_per_token": (gamma * t_draft + t_verify) / om}
    return out


def load_traffic(name):
    """DRAM bytes per verify launch from the committed ncu summary; None once the kernel source changed."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "verify_attention_traffic.json")
    src = os.path.join(ROOT, "long_context_speculative_split_gb300", "csrc", "attn_tc.cu")
    try:
        with open(path) as f:
            d = json.load(f)
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        if d.get("kernel_source_sha256_16") != sha:
            return None
        return d.get(name)
    except Exception:
        return None


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_ranks(args.gpus, argv)  # one rank per GPU, each runs the rest of main()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "round_b32_ctx16k_32layers":
        return run_round(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
