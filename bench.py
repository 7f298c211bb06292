#!/usr/bin/env python
"""Drafter-cycle benchmark: inject + draft block + top-K + DDTree build.

One step is one drafter cycle of the Qwen3-8B-shaped batch-1 workload
(5 layers, hidden 4096, 32/8 heads of 128, FFN 12288, vocabulary 151936,
8192 injected context positions, block L = 16, top-K 8, DDTree budget 256):
  dflash_draft_cycle  dflash_inject_kv (the 16 newest context positions: W_proj
                      and U_K/U_V) then dflash_draft_block (5 layers + LM head +
                      log-softmax + top-K), one call
  ddtree_build        Algorithm 1 + ancestor mask
The acceptance walk is timed separately (accept_us).  Inputs are seeded
synthetic data of those shapes (no trained weights or datasets exist here).

Timed region: K replays of a CUDA graph of the cycle, CUDA events on the
launching stream, barrier + synchronize on both sides, max over ranks.  Each
cycle streams ~3.6 GB of weights and cache, far above the 129 MB L2, so no
flush is needed between steps.  Per-kernel times (roofline, shares) come from
traced eager cycles: CUDA events recorded around every kernel launch through
the library's trace hook, queued behind a GPU sleep so that host latency does
not leak into them (they run without the graph's launch overlap).  e2e repeats the cycle through the C-ABI calls with
pinned host inputs and outputs, copies included.

--impl reference times the CPU oracle on the same workload (bounded sample).
Multi-GPU (torchrun): every rank runs an independent replica (batch-1 drafting
does not shard); value is the sum of cycles/s over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "draft cycles/sec & µs/cycle (inject+draft+top-K+DDTree) at Qwen3-8B shape"
UNIT = "cycles/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' sub-records")
    ap.add_argument("--cpu-budget-s", type=float, default=60.0)
    ap.add_argument("--oracle-cycle-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--topk-rows", type=int, default=0,
                    help="topk_stress: time only the first N rows (a smaller profiling case)")
    ap.add_argument("--case", choices=["lm_head_gemm", "down_gemm", "o_gemm", "gate_up_gemm_b32",
                                       "lm_head_gemm_b32", "o_gemm_b32", "topk_stress",
                                       "topk_b1", "tree_stress", "tree_b1", "tree_attention",
                                       "chain_sweep", "budget_sweep", "steady_state"],
                    default=None, help="time one kernel alone (microbenchmark / ncu target)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: barrier and max-over-ranks timing)
# ---------------------------------------------------------------------------

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(ms_step_max: float, world: int) -> float:
    """Whole-job cycles/s of `world` independent replicas (one cycle per rank
    per step), timed by the slowest rank: weak scaling."""
    return world * 1e3 / ms_step_max


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        bus = None
        try:
            p = torch.cuda.get_device_properties(torch.cuda.current_device())
            bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            pass
        rows = [l.split(", ") for l in self.lines if l]
        rows = [r for r in rows if len(r) >= 10]
        if bus is not None:
            mine = [r for r in rows if r[1].upper().endswith(bus[-12:])]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# workload set-up (untimed)
# ---------------------------------------------------------------------------

def gemm_shapes(s, M_inject, R):
    """(name, M, N, K) of every tensor-core GEMM of one cycle."""
    out = [("w_proj", M_inject, s.d, s.n_feat * s.d_feat),
           ("u_kv", M_inject, s.n_layers * 2 * s.kv_dim, s.d)]
    for _ in range(s.n_layers):
        out += [("qkv", R, s.qkv_dim, s.d), ("o", R, s.d, s.n_q * s.head_dim),
                ("gate_up", R, 2 * s.d_ff, s.d), ("down", R, s.d, s.d_ff)]
    out.append(("lm_head", R, s.vocab, s.d))
    return out


def algorithmic_bytes(s, wl, ctx):
    """Bytes one cycle must move at least: every weight once, the context KV once,
    the logits written and read once, the new features read once."""
    es = 2 if s.dtype == "bf16" else 4
    R = wl.n_req * wl.L
    w = sum(N * K for _, _, N, K in gemm_shapes(s, wl.n_req * wl.L, R)) * es
    kv = int(np.sum(ctx)) * s.n_layers * 2 * s.kv_dim * es
    logits = 2 * wl.n_req * (wl.L - 1) * s.vocab * 4
    feats = wl.n_req * wl.L * s.n_feat * s.d_feat * es
    return w + kv + logits + feats, w


class Cycle:
    def __init__(self, wid):
        from block_diffusion_speculative_kv_gb300 import binding as bd
        from block_diffusion_speculative_kv_gb300 import synth
        from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
        from block_diffusion_speculative_kv_gb300.drafter import Drafter
        self.bd = bd
        self.wl_id = wid
        self.wl = wl = WORKLOADS[wid]
        self.s = s = wl.shape
        dev = "cuda"
        self.ctx = synth.context_lengths(wl)
        T = int(self.ctx.max())
        L, n_req = wl.L, wl.n_req
        self.w = synth.drafter_weights(s, wl.seed, device=dev)
        prefill_rows = int(np.sum(self.ctx - L))
        self.dr = Drafter(s, self.w, n_req=n_req, cap=wl.cap,
                          max_inject_rows=max(prefill_rows, n_req * L), L=L, K=wl.K)
        i32 = dict(dtype=torch.int32, device=dev)
        # untimed prefill: context [0, T-L) of every request from N(0,1) features
        rows = (self.ctx - L).astype(np.int64)
        off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
        feats = synth.features(int(off[-1]), s, wl.seed, stream=101, device=dev)
        self.dr.inject_kv(feats, torch.as_tensor(off, **i32),
                          torch.zeros(n_req, **i32))
        del feats
        # per-cycle inputs: the L newest positions [ctx-L, ctx) of each request
        self.feats = synth.features(n_req * L, s, wl.seed, stream=102, device=dev)
        self.row_off = torch.as_tensor(np.arange(n_req + 1, dtype=np.int32) * L, **i32)
        self.pos0 = torch.as_tensor(self.ctx - L, **i32)
        self.ctx_len = torch.as_tensor(self.ctx, **i32)
        self.anchor = torch.as_tensor(synth.anchors(n_req, s.vocab, s.mask_id, wl.seed), **i32)
        self.max_ctx = T
        D = L - 1
        self.ids = torch.empty(n_req, D, wl.K, **i32)
        self.lp = torch.empty(n_req, D, wl.K, dtype=torch.float32, device=dev)
        self.tree = bd.tree_buffers(n_req, wl.B, dev)
        self.accept_len = torch.empty(n_req, **i32)
        self.accepted = torch.empty(n_req, D, **i32)
        self.bonus = torch.empty(n_req, **i32)
        torch.cuda.synchronize()
        self.target = None

    def run(self, sampling=None):
        # inject + draft as one C-ABI call (the injection's GEMMs share a
        # launch with the first QKV projection), then the tree
        self.dr.draft_cycle(self.feats, self.row_off, self.pos0, self.anchor, self.ctx_len,
                            self.max_ctx, self.ids, self.lp, sampling=sampling)
        self.bd.ddtree_build(self.lp, self.ids, self.anchor, self.wl.B, *self.tree)

    def make_targets(self):
        from block_diffusion_speculative_kv_gb300 import synth
        torch.cuda.synchronize()
        n_nodes = self.tree[0].cpu().numpy()
        depth = self.tree[3].cpu().numpy()
        tgt = synth.target_tokens(n_nodes, depth, self.lp.cpu().numpy(), self.ids.cpu().numpy(),
                                  self.s.vocab, self.wl.target_agree, seed=self.wl.seed)
        self.target = torch.as_tensor(tgt, device="cuda")

    def accept(self):
        self.bd.ddtree_accept(self.wl.L - 1, self.wl.B, self.tree[0], self.tree[1], self.tree[2],
                              self.target, self.accept_len, self.accepted, self.bonus)


class Tracer:
    """Records CUDA events around every library kernel launch."""

    def __init__(self):
        self.open = []
        self.done = []

    def __call__(self, name, phase, stream):
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(torch.cuda.current_stream())
        if phase == 0:
            self.open.append((name, ev))
        else:
            n, e0 = self.open.pop()
            self.done.append((n, e0, ev))

    def durations(self):
        torch.cuda.synchronize()
        out = {}
        for n, e0, e1 in self.done:
            out.setdefault(n, []).append(e0.elapsed_time(e1) * 1e3)   # us
        return out


def timed_region(fn, steps, warmup, world):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    clk = ClockSampler()
    clk.start()
    time.sleep(0.3)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(steps):
        fn()
    e1.record(st)
    torch.cuda.synchronize()
    barrier(world)
    clk.stop()
    return e0.elapsed_time(e1), clk.summary()


def traffic_from_profile(kernel_src):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary,
    only if the kernel source is unchanged since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_qwen3_8b_b1.md")
    if not os.path.exists(path):
        return None
    sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    meta = {}
    for line in open(path):
        if line.startswith("<!-- ") and ":" in line:
            k, v = line[5:].split("-->")[0].split(":", 1)
            meta[k.strip()] = v.strip()
    if meta.get("kernel_sha") != sha:
        return None
    try:
        return float(meta["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class HostCycle:
    """One request's cycle of a workload, as host arrays for the oracle.

    Nothing here touches the CUDA library: the weights are either drawn on
    the host from the workload's seed or copied from tensors the caller
    already holds, the context cache [0, T) is a seeded N(0, 1) prefix (the
    same distribution an injected context has), and the cycle's L newest
    feature rows are drawn on the host."""

    def __init__(self, wid, weights=None):
        from block_diffusion_speculative_kv_gb300 import synth
        from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
        self.wl = wl = WORKLOADS[wid]
        self.s = s = wl.shape
        w = weights if weights is not None else synth.drafter_weights(s, wl.seed, device="cpu")
        self.w = {k: ([_F64(t) for t in v] if isinstance(v, list) else _F64(v))
                  for k, v in w.items()}
        self.T = int(synth.context_lengths(wl)[0])
        ks, vs = synth.cache_prefix(s, 1, self.T, wl.seed, device="cpu")
        self.ck = [_F64(k[0]) for k in ks]
        self.cv = [_F64(v[0]) for v in vs]
        self.feats = _F64(synth.features(wl.L, s, wl.seed, stream=102, device="cpu"))
        self.anchor = int(synth.anchors(1, s.vocab, s.mask_id, wl.seed)[0])
        self.dims = dict(n_layers=s.n_layers, d=s.d, n_q=s.n_q, n_kv=s.n_kv,
                         head_dim=s.head_dim, vocab=s.vocab, mask_id=s.mask_id,
                         rope_theta=s.rope_theta, rms_eps=s.rms_eps)

    def run(self):
        """One oracle cycle: inject the L newest rows, the block pass, log-softmax
        and top-K, Algorithm 1.  Returns its wall time in seconds."""
        from oracle import ddtree as odt
        from oracle import drafter as od
        s, wl = self.s, self.wl
        t0 = time.perf_counter()
        f = od.fuse_features(self.feats, self.w["w_proj"])
        pos = self.T - wl.L + np.arange(wl.L)
        for l in range(s.n_layers):
            od.inject_kv(f, self.w["uk"][l], self.w["uv"][l], pos, s.n_kv, s.head_dim,
                         s.rope_theta)
        logits = od.drafter_block(self.w, self.dims, self.ck, self.cv, self.T, self.anchor,
                                  wl.L)
        ids, lp, _ = od.logits_topk(logits, wl.K)
        odt.build_tree(lp.astype(np.float32), ids, self.anchor, wl.B)
        return time.perf_counter() - t0


class _F64:
    """Lazy float64 view of a host tensor (bf16 has no NumPy dtype)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, i):
        return self.t[i].float().numpy().astype(np.float64)

    def __array__(self, dtype=None, copy=None):
        return self.t.float().numpy().astype(np.float64)


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


SAMPLE_TEXT = ("one full oracle cycle of request 0 (inject of the L newest rows, every layer "
               "over the whole context, LM head over the vocabulary, top-K, Algorithm 1), "
               "NumPy float64; inputs built on the host (context cache: seeded N(0,1) prefix)")


def one_core_oracle(wid, timeout_s=600):
    """The same oracle cycle pinned to one core, in a child process whose BLAS
    thread count is fixed before NumPy loads.  Returns seconds or an error."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-cycle-child", "--workload",
           str(wid)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=timeout_s)
    except subprocess.TimeoutExpired:
        return {"error": f"over {timeout_s} s"}
    for line in r.stdout.splitlines()[::-1]:
        if line.startswith("{"):
            return json.loads(line)
    return {"error": (r.stderr or r.stdout)[-300:]}


def oracle_cycle_child(wid):
    """Entry of the one-core child: pin to one core, time one oracle cycle."""
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except (AttributeError, OSError):
        pass
    torch.set_num_threads(1)
    hc = HostCycle(wid)
    dt = hc.run()
    print(json.dumps({"seconds": dt, "cores": _cores()}))


def cpu_baseline(cyc, budget_s):
    """Time the CPU oracle on one request's cycle on this host's cores (all of
    them, then one), with the bench's weights copied to the host and the rest
    of the inputs built there."""
    hc = HostCycle(cyc.wl_id, weights={k: ([t.cpu() for t in v] if isinstance(v, list)
                                          else v.cpu()) for k, v in cyc.w.items()})
    dt = hc.run()
    one = one_core_oracle(cyc.wl_id, timeout_s=max(60.0, 10 * budget_s))
    out = {"value": 1.0 / dt, "unit": UNIT, "cores": _cores(), "kind": "oracle",
           "sample": SAMPLE_TEXT + "; %.1f s on all cores" % dt}
    if "seconds" in one:
        out["one_core"] = {"value": 1.0 / one["seconds"], "unit": UNIT, "cores": one["cores"],
                           "seconds": round(one["seconds"], 2)}
    else:
        out["one_core"] = {"value": None, "error": one.get("error")}
    return out


def run_reference(args, rank, world):
    """The oracle arm: full oracle cycles on the host cores, inputs built on
    the host (the CUDA library is never loaded)."""
    if rank != 0:
        return
    hc = HostCycle(args.workload)
    times = []
    t_start = time.perf_counter()
    steps_done = 0
    warm = max(args.warmup, 3)
    for i in range(warm + args.steps):
        dt = hc.run()
        if i >= warm:
            times.append(dt)
            steps_done += 1
        if time.perf_counter() - t_start > 240 and steps_done >= 1:
            break
    ms = 1e3 * statistics.mean(times)
    val = 1e3 / ms
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1,
            "steps": steps_done, "warmup": warm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": hc.wl.name},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": SAMPLE_TEXT + "; steps capped to end within a few "
                                                     "minutes"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def graph_time(fn, steps, warmup):
    """Milliseconds for `steps` replays of a CUDA graph of fn (host launch cost
    out of the timed region), and the clock record."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return timed_region(g.replay, steps, warmup, 1)


def traced_us(fn, reps=3):
    """Per-kernel microseconds of one call of fn (CUDA events around each of
    the library's launches, the host queue filled ahead by a GPU-side sleep)."""
    from block_diffusion_speculative_kv_gb300 import binding as bd
    tr = Tracer()
    for _ in range(reps):
        torch.cuda._sleep(20_000_000)
        bd.set_trace_hook(tr)
        fn()
        bd.set_trace_hook(None)
    return {k: round(sum(v) / reps, 2) for k, v in tr.durations().items()}


def run_chain_sweep(args):
    """Vanilla DFlash (a chain of the per-position argmax at T = 0, or of one
    Gumbel-max sample per position at T = 1, drafted inside the LM-head top-K
    pass) against DDTree (top-8 per position, budget B) at block sizes L = 4,
    8, 16, on the Qwen3-8B-shaped batch-1 drafter with 8192 context slots.
    One line per (drafter, L, T): microseconds per draft cycle (inject + draft
    + tree) as CUDA-graph replays, and the kernels' times in one traced cycle."""
    cyc = Cycle(2)
    bd = cyc.bd
    wl = cyc.wl
    i32 = dict(dtype=torch.int32, device="cuda")
    rows = []
    for L in (4, 8, 16):
        D = L - 1
        feats = cyc.feats[:L].contiguous()
        row_off = torch.tensor([0, L], **i32)
        pos0 = torch.as_tensor(cyc.ctx - L, **i32)
        for drafter, T in (("chain", 0.0), ("chain", 1.0), ("ddtree", 0.0)):
            K = 1 if drafter == "chain" else wl.K
            B = D if drafter == "chain" else wl.B
            ids = torch.empty(1, D, K, **i32)
            lq = torch.empty(1, D, K, dtype=torch.float32, device="cuda")
            tree = bd.tree_buffers(1, B, "cuda")
            smp = (T, 12345, 0) if T > 0 else None

            def fn():
                cyc.dr.draft_cycle(feats, row_off, pos0, cyc.anchor, cyc.ctx_len, cyc.max_ctx,
                                   ids, lq, L=L, K=K, sampling=smp)
                if drafter == "chain":
                    bd.chain_tree(ids, cyc.anchor, B, *tree)
                else:
                    bd.ddtree_build(lq, ids, cyc.anchor, B, *tree)
            ms, clocks = graph_time(fn, args.steps, max(args.warmup, 3))
            assert cyc.dr.read_status() == 0
            rows.append({"drafter": drafter, "L": L, "T": T, "K": K, "B": B,
                         "us_per_cycle": round(ms * 1e3 / args.steps, 1),
                         "kernels_us": traced_us(fn),
                         "sm_mhz": clocks.get("sm_mhz") if isinstance(clocks, dict) else None})
    print(json.dumps({"case": "chain_sweep", "workload": wl.name, "steps": args.steps,
                      "rows": rows}))


def run_budget_sweep(args):
    """DDTree node budget B = 16 .. 1024 on the Qwen3-8B-shaped batch-1 drafter
    (8192 context slots), with the workload's K = 8 and with Lemma 1's exact
    K = B.  Per (B, K): microseconds per full cycle (inject + draft + top-K +
    tree), for the top-K alone over the cycle's 15 rows of fp32 logits, and for
    the tree build alone (kernel times from CUDA events around each launch; the
    cycle as CUDA-graph replays); the tree's node count and depth."""
    cyc = Cycle(2)
    bd, wl = cyc.bd, cyc.wl
    L, D = wl.L, wl.L - 1
    i32 = dict(dtype=torch.int32, device="cuda")
    nbytes = int(bd.lib().dflash_workspace_bytes(cyc.dr.handle, 1, L, L, 1024))
    cyc.dr.ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    logits = torch.empty(1, D, wl.shape.vocab, dtype=torch.float32, device="cuda")
    cyc.dr.draft_cycle(cyc.feats, cyc.row_off, cyc.pos0, cyc.anchor, cyc.ctx_len, cyc.max_ctx,
                       cyc.ids, cyc.lp, logits)
    lg2 = logits.reshape(D, wl.shape.vocab)
    rows = []
    for B in (16, 32, 64, 128, 256, 512, 1024):
        for K in sorted({wl.K, B}):
            ids = torch.empty(1, D, K, **i32)
            lq = torch.empty(1, D, K, dtype=torch.float32, device="cuda")
            tree = bd.tree_buffers(1, B, "cuda")
            tws = torch.zeros(bd.topk_workspace_bytes(D, wl.shape.vocab, K), dtype=torch.uint8,
                              device="cuda")

            def cycle_fn():
                cyc.dr.draft_cycle(cyc.feats, cyc.row_off, cyc.pos0, cyc.anchor, cyc.ctx_len,
                                   cyc.max_ctx, ids, lq, K=K)
                bd.ddtree_build(lq, ids, cyc.anchor, B, *tree)

            def topk_fn():
                bd.logits_topk(lg2, K, ids.reshape(D, K), lq.reshape(D, K), tws)

            def tree_fn():
                bd.ddtree_build(lq, ids, cyc.anchor, B, *tree)
            w = max(args.warmup, 3)
            ms_c, clocks = graph_time(cycle_fn, args.steps, w)
            tk = traced_us(topk_fn)
            tt = traced_us(tree_fn)
            assert cyc.dr.read_status() == 0
            rows.append({"B": B, "K": K, "us_cycle": round(ms_c * 1e3 / args.steps, 1),
                         "cycle_kernels_us": traced_us(cycle_fn),
                         "us_topk": round(sum(tk.values()), 2), "topk_kernels_us": tk,
                         "us_tree": round(sum(tt.values()), 2),
                         "n_nodes": int(tree[0].item()), "depth": int(tree[3].max().item()),
                         "max_rank": int(tree[4].max().item()),
                         "sm_mhz": clocks.get("sm_mhz") if isinstance(clocks, dict) else None})
    print(json.dumps({"case": "budget_sweep", "workload": wl.name, "steps": args.steps,
                      "rows": rows}))


def run_steady_state(args):
    """Chained cycles on the device at the Qwen3-8B batch-1 shape: each cycle
    injects the previous cycle's accepted path (dflash_draft_cycle with the
    rows, positions and features dflash_commit_accepted wrote), drafts from the
    bonus token, builds the tree (B = 256), walks it against a device-side
    stand-in for the target's choices, and commits.  One captured CUDA graph
    of a cycle replayed `steps` times; the context grows by tau per cycle."""
    from block_diffusion_speculative_kv_gb300 import binding as bd
    from block_diffusion_speculative_kv_gb300 import synth
    from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
    from block_diffusion_speculative_kv_gb300.drafter import Drafter
    torch.cuda.set_device(0)
    wl = WORKLOADS[2]
    s = wl.shape
    L, D, B = wl.L, wl.L - 1, wl.B
    n_cycles = args.steps + max(args.warmup, 3) + 3
    ctx0 = int(wl.ctx[1])
    cap = ctx0 + (n_cycles + 2) * L
    w = synth.drafter_weights(s, wl.seed, device="cuda")
    dr = Drafter(s, w, n_req=1, cap=cap, max_inject_rows=ctx0, L=L, K=wl.K)
    fd = s.n_feat * s.d_feat
    i32 = dict(dtype=torch.int32, device="cuda")
    pre = synth.features(ctx0, s, wl.seed, stream=101, device="cuda")
    dr.inject_kv(pre[:ctx0 - L], torch.tensor([0, ctx0 - L], **i32), torch.zeros(1, **i32))
    feats = pre[ctx0 - L:].contiguous()
    del pre
    tree_feats = synth.features(B + 1, s, wl.seed, stream=103, device="cuda").reshape(1, B + 1, fd)
    row_off = torch.tensor([0, L], **i32)
    pos0 = torch.tensor([ctx0 - L], **i32)
    ctx_len = torch.tensor([ctx0], **i32)
    anchor = torch.as_tensor(synth.anchors(1, s.vocab, s.mask_id, wl.seed), **i32)
    ids = torch.empty(1, D, wl.K, **i32)
    lp = torch.empty(1, D, wl.K, dtype=torch.float32, device="cuda")
    tree = bd.tree_buffers(1, B, "cuda")
    al, acc, bonus = torch.empty(1, **i32), torch.empty(1, D, **i32), torch.empty(1, **i32)
    taus = torch.zeros(1, dtype=torch.int64, device="cuda")

    def cycle():
        dr.draft_cycle(feats, row_off, pos0, anchor, ctx_len, cap, ids, lp)
        bd.ddtree_build(lp, ids, anchor, B, *tree)
        target = synth.target_first_child(tree[0], tree[1], tree[2], s.vocab)
        bd.ddtree_accept(D, B, tree[0], tree[1], tree[2], target, al, acc, bonus)
        bd.commit_accepted(D, tree_feats, al, acc, bonus, ctx_len, anchor, row_off, pos0, feats)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cycle()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cycle()
    torch.cuda.synchronize()
    c0 = int(ctx_len.item())
    ms, clocks = timed_region(g.replay, args.steps, max(args.warmup, 3), 1)
    c1 = int(ctx_len.item())
    assert dr.read_status() == 0
    cycles = args.steps + max(args.warmup, 3)
    us = ms * 1e3 / args.steps
    print(json.dumps({"case": "steady_state", "workload": wl.name, "cycles": cycles,
                      "us_per_cycle": round(us, 1), "mean_tau": round((c1 - c0) / cycles, 3),
                      "tokens_per_s_drafter_side": round((c1 - c0) / cycles / (us * 1e-6), 1),
                      "ctx_start": c0, "ctx_end": c1, "clocks": clocks,
                      "timed": "CUDA graph of one cycle (draft_cycle + ddtree_build + target "
                               "stand-in + ddtree_accept + commit), replayed"}))


def run_case(args):
    """One kernel on its own, launched back to back (inputs larger than L2)."""
    if args.case == "steady_state":
        return run_steady_state(args)
    if args.case == "chain_sweep":
        return run_chain_sweep(args)
    if args.case == "budget_sweep":
        return run_budget_sweep(args)
    from block_diffusion_speculative_kv_gb300 import binding as bd
    from block_diffusion_speculative_kv_gb300 import synth
    from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda").manual_seed(1)
    if args.case in ("lm_head_gemm", "down_gemm", "o_gemm", "gate_up_gemm_b32",
                     "lm_head_gemm_b32", "o_gemm_b32"):
        # batch 1 (16 rows) and the 32-request batch (512 rows) of the
        # Qwen3-8B-shaped drafter
        M, N, K = {"lm_head_gemm": (16, 151936, 4096), "down_gemm": (16, 4096, 12288),
                   "o_gemm": (16, 4096, 4096), "gate_up_gemm_b32": (512, 24576, 4096),
                   "lm_head_gemm_b32": (480, 151936, 4096),
                   "o_gemm_b32": (512, 4096, 4096)}[args.case]
        copies = max(1, int(math.ceil(400e6 / (2 * N * K))))   # rotate > L2 of weights
        X = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
        Ws = [torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
              for _ in range(copies)]
        Y = torch.empty(M, N, device="cuda")
        ws = torch.zeros(bd.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        fn_i = [0]

        def fn():
            bd.linear_bf16(X, Ws[fn_i[0] % copies], Y, ws)
            fn_i[0] += 1
        nbytes = 2 * N * K + 2 * M * K + 4 * M * N
    elif args.case in ("topk_stress", "topk_b1"):
        wl = WORKLOADS[4]
        logits, _ = synth.stress_logits(wl.n_req, wl.D, wl.vocab, wl.seed, device="cuda")
        if args.case == "topk_b1":   # the 8B batch-1 drafter's 15 rows of fp32 logits
            logits = logits[:15].float().contiguous()
        elif args.topk_rows:
            logits = logits[:args.topk_rows].contiguous()
        rows = logits.shape[0]
        ids = torch.empty(rows, wl.K, dtype=torch.int32, device="cuda")
        lp = torch.empty(rows, wl.K, device="cuda")
        ws = torch.zeros(bd.topk_workspace_bytes(rows, wl.vocab, wl.K), dtype=torch.uint8,
                         device="cuda")

        def fn():
            bd.logits_topk(logits, wl.K, ids, lp, ws)
        nbytes = logits.numel() * 2
    elif args.case == "tree_attention":
        # one Qwen3-8B-shaped target layer of the verification pass: 32/8 heads
        # of 128, 8192 context slots, the 257-node tree of the batch-1 workload
        wl = WORKLOADS[2]
        n_q, n_kv, hd, B, T = 32, 8, 128, wl.B, 8192
        lp, idt = synth.random_topk_table(1, wl.D, wl.K, 151936, wl.seed)
        bufs = bd.tree_buffers(1, B, "cuda")
        bd.ddtree_build(torch.from_numpy(lp).cuda(), torch.from_numpy(idt).cuda(),
                        torch.zeros(1, dtype=torch.int32, device="cuda"), B, *bufs)
        n_nodes, mask = bufs[0], bufs[5]
        copies = 5                                    # 5 x 33.5 MB of cache > L2
        cks = [(torch.randn(1, n_kv, T, hd, generator=g, device="cuda") * 0.35).to(torch.bfloat16)
               for _ in range(copies)]
        cvs = [torch.randn(1, n_kv, T, hd, generator=g, device="cuda").to(torch.bfloat16)
               for _ in range(copies)]
        q = (torch.randn(1, B + 1, n_q * hd, generator=g, device="cuda") * 0.35).to(torch.bfloat16)
        k = (torch.randn(1, B + 1, n_kv * hd, generator=g, device="cuda") * 0.35).to(torch.bfloat16)
        v = torch.randn(1, B + 1, n_kv * hd, generator=g, device="cuda").to(torch.bfloat16)
        out = torch.empty_like(q)
        ctx = torch.full((1,), T, dtype=torch.int32, device="cuda")
        ws = torch.zeros(bd.tree_attention_workspace_bytes(1, n_q, n_kv, hd, B, T),
                         dtype=torch.uint8, device="cuda")
        fn_i = [0]

        def fn():
            c = fn_i[0] % copies
            bd.tree_attention(q, k, v, cks[c], cvs[c], ctx, T, mask, n_nodes, out, ws)
            fn_i[0] += 1
        torch.cuda.synchronize()
        nn = int(n_nodes.item())
        d_cpu = bufs[3].cpu().numpy()[0]
        anc = int(sum(int(d_cpu[i]) + 1 for i in range(nn + 1)))   # |ancestors incl. self|
        flops = 4.0 * hd * n_q * ((nn + 1) * T + anc)
        nbytes = 2 * 2 * n_kv * T * hd + 3 * 2 * (B + 1) * n_q * hd
    else:
        wl = WORKLOADS[4] if args.case == "tree_stress" else WORKLOADS[2]
        lp, idt = synth.random_topk_table(wl.n_req, wl.D, wl.K, 151936, wl.seed)
        lp_d, id_d = torch.from_numpy(lp).cuda(), torch.from_numpy(idt).cuda()
        roots = torch.zeros(wl.n_req, dtype=torch.int32, device="cuda")
        bufs = bd.tree_buffers(wl.n_req, wl.B, "cuda")

        def fn():
            bd.ddtree_build(lp_d, id_d, roots, wl.B, *bufs)
        nbytes = 0
    ms, clocks = timed_region(fn, args.steps, max(args.warmup, 3), 1)
    us = ms * 1e3 / args.steps
    out = {"case": args.case, "us_per_launch": round(us, 2), "steps": args.steps,
           "clocks": clocks}
    if nbytes:
        out["gbs"] = round(nbytes / (us * 1e-6) / 1e9, 1)
    if args.case.endswith("_gemm") or args.case.endswith("_b32"):
        if args.case.startswith(("lm_head", "down", "o_", "gate_up")):
            out["tflops"] = round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1)
    if args.case == "tree_attention":
        out["tflops"] = round(flops / (us * 1e-6) / 1e12, 1)
        out["nodes"] = nn + 1
    print(json.dumps(out))


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        pk = json.load(open(path))
        return (float(pk["hbm_gbs"]), float(pk["bf16_tflops"]),
                float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def gemm_flops_algorithmic(s, wl):
    """FLOPs of one cycle's GEMMs that the method needs: every projection over
    the n_req*L block rows, the LM head over the n_req*(L-1) drafted rows."""
    R = wl.n_req * wl.L
    f = 0
    for name, M, N, K in gemm_shapes(s, R, R):
        f += 2 * (wl.n_req * (wl.L - 1) if name == "lm_head" else M) * N * K
    return f


def sub_cycle_record(wid, steps, warmup, sampling=None, cyc=None):
    """One more workload's drafter cycle (CUDA-graph replays) with its roofline.
    With `sampling` = (T, seed) the cycle is vanilla DFlash drafting at
    temperature T: one Gumbel-max draw per block position inside the LM-head
    pass, laid out as a chain (DDTree's own tree does not depend on T: the
    temperature only changes how the target picks its tokens)."""
    hbm, tc, tc_sus, src = _peaks()
    own = cyc is None
    if own:
        cyc = Cycle(wid)
    s, wl = cyc.s, cyc.wl
    if sampling:
        bd = cyc.bd
        D = wl.L - 1
        i32 = dict(dtype=torch.int32, device="cuda")
        c_ids = torch.empty(wl.n_req, D, 1, **i32)
        c_lq = torch.empty(wl.n_req, D, 1, dtype=torch.float32, device="cuda")
        c_tree = bd.tree_buffers(wl.n_req, D, "cuda")

        def fn():
            cyc.dr.draft_cycle(cyc.feats, cyc.row_off, cyc.pos0, cyc.anchor, cyc.ctx_len,
                               cyc.max_ctx, c_ids, c_lq, K=1, sampling=sampling)
            bd.chain_tree(c_ids, cyc.anchor, D, *c_tree)
    else:
        fn = cyc.run
    ms, clocks = graph_time(fn, steps, warmup)
    us = ms * 1e3 / steps
    if cyc.dr.read_status() != 0:
        raise RuntimeError("device status after the timed cycles")
    kern = traced_us(fn)
    nbytes, _ = algorithmic_bytes(s, wl, cyc.ctx)
    rec = {"workload": wl.name, "n_req": wl.n_req, "us_per_cycle": round(us, 1),
           "cycles_per_s": round(1e6 / us, 2), "request_drafts_per_s": round(wl.n_req * 1e6 / us, 1),
           "cycle_hbm": {"algorithmic_bytes": int(nbytes),
                         "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                         "frac": round(nbytes / (us * 1e-6) / 1e9 / hbm, 4)},
           "kernel_us_per_cycle": kern, "clocks": clocks,
           "timed": "CUDA graph of inject + draft + top-K + DDTree build, replayed"}
    if sampling:
        rec["sampling"] = {"temperature": sampling[0], "seed": sampling[1],
                           "drafter": "vanilla DFlash chain, K = 1 Gumbel-max draw per position"}
        rec["timed"] = "CUDA graph of inject + draft + sampling + chain tree, replayed"
    if wl.n_req > 1:
        flops = gemm_flops_algorithmic(s, wl)
        g_us = kern.get("gemm_tc", float("nan"))
        tfl = flops / (g_us * 1e-6) / 1e12
        rec["gemm"] = {"bound": "tensor", "kernel": "gemm_tc", "flops_per_cycle": int(flops),
                       "us_per_cycle": g_us, "achieved": round(tfl, 1), "unit": "TFLOP/s",
                       "peak": tc_sus, "peak_source": src + " (sustained: the GEMMs run inside "
                                                             "a multi-ms cycle)",
                       "frac": round(tfl / tc_sus, 4), "frac_of_burst": round(tfl / tc, 4)}
        a_us = kern.get("attn_split", 0.0) + kern.get("attn_combine", 0.0)
        kv = int(np.sum(cyc.ctx)) * s.n_layers * 2 * s.kv_dim * 2
        if a_us > 0:
            rec["attention"] = {"kv_bytes_per_cycle": kv, "us_per_cycle": round(a_us, 1),
                                "achieved_gbs": round(kv / (a_us * 1e-6) / 1e9, 1),
                                "frac": round(kv / (a_us * 1e-6) / 1e9 / hbm, 4)}
    if own:
        cyc.dr.close()
        del cyc
        torch.cuda.empty_cache()
    return rec


def stress_record(steps, warmup):
    """The top-K + tree stress workload: 256 requests x 16 positions x 151936 bf16
    logits, top-8 per row (HBM-bound read), then a B = 512 tree per request."""
    from block_diffusion_speculative_kv_gb300 import binding as bd
    from block_diffusion_speculative_kv_gb300 import synth
    from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
    hbm, _, _, src = _peaks()
    wl = WORKLOADS[4]
    logits, _ = synth.stress_logits(wl.n_req, wl.D, wl.vocab, wl.seed, device="cuda")
    rows = logits.shape[0]
    ids = torch.empty(rows, wl.K, dtype=torch.int32, device="cuda")
    lp = torch.empty(rows, wl.K, device="cuda")
    ws = torch.zeros(bd.topk_workspace_bytes(rows, wl.vocab, wl.K), dtype=torch.uint8,
                     device="cuda")
    ms_t, clk_t = timed_region(lambda: bd.logits_topk(logits, wl.K, ids, lp, ws), steps, warmup, 1)
    us_t = ms_t * 1e3 / steps
    nbytes = logits.numel() * logits.element_size()
    gbs = nbytes / (us_t * 1e-6) / 1e9
    lp3 = lp.reshape(wl.n_req, wl.D, wl.K)
    id3 = ids.reshape(wl.n_req, wl.D, wl.K)
    roots = torch.zeros(wl.n_req, dtype=torch.int32, device="cuda")
    bufs = bd.tree_buffers(wl.n_req, wl.B, "cuda")
    ms_b, _ = timed_region(lambda: bd.ddtree_build(lp3, id3, roots, wl.B, *bufs), steps, warmup, 1)
    if bd.read_status(ws) != 0:
        raise RuntimeError("device status after the stress top-K")
    rec = {"workload": wl.name, "rows": rows, "vocab": wl.vocab, "K": wl.K, "B": wl.B,
           "topk": {"us_per_launch": round(us_t, 2), "bytes": int(nbytes),
                    "achieved_gbs": round(gbs, 1), "peak": hbm, "peak_source": src,
                    "frac": round(gbs / hbm, 4), "clocks": clk_t,
                    "l2": "1.245 GB of logits per launch, larger than L2"},
           "tree_us_per_launch": round(ms_b * 1e3 / steps, 2),
           "tree_nodes_mean": round(float(bufs[0].float().mean().item()), 1)}
    del logits
    torch.cuda.empty_cache()
    return rec


def main():
    args = parse()
    if args.oracle_cycle_child:
        oracle_cycle_child(args.workload)
        return
    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        # host-only: rank 0 times the oracle, other ranks exit without work
        run_reference(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_init()
    from block_diffusion_speculative_kv_gb300 import binding as bd
    cyc = Cycle(args.workload)
    s, wl = cyc.s, cyc.wl

    # ---- launches per cycle (trace hook, eager) ----
    count = [0]

    def counter(name, phase, stream):
        if phase == 0:
            count[0] += 1

    bd.set_trace_hook(counter)
    cyc.run()
    bd.set_trace_hook(None)
    launches_per_cycle = count[0]
    torch.cuda.synchronize()
    cyc.make_targets()

    # ---- graph of one cycle ----
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            cyc.run()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cyc.run()
    torch.cuda.synchronize()

    ms_total, clocks = timed_region(graph.replay, args.steps, max(args.warmup, 3), world)
    ms_step = max_over_ranks(ms_total / args.steps, world)
    status = cyc.dr.read_status()
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")

    # ---- per-kernel times from traced eager cycles ----
    # a GPU-side sleep ahead of each traced cycle lets the host queue every
    # launch (and its events) before the GPU reaches them, so the events time
    # the kernels and not the host callbacks in between
    tr = Tracer()
    for _ in range(3):
        torch.cuda._sleep(20_000_000)
        bd.set_trace_hook(tr)
        cyc.run()
        bd.set_trace_hook(None)
    dur = tr.durations()
    per_cycle = {k: sum(v) / 3.0 for k, v in dur.items()}
    launches = {k: len(v) // 3 for k, v in dur.items()}
    total_k = sum(per_cycle.values())
    shares = {k: round(v / total_k, 4) for k, v in sorted(per_cycle.items(), key=lambda x: -x[1])}

    # ---- acceptance walk on its own ----
    for _ in range(3):
        cyc.accept()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(20):
        cyc.accept()
    a1.record()
    torch.cuda.synchronize()
    accept_us = a0.elapsed_time(a1) * 1e3 / 20

    # ---- roofline of the dominant kernel (the tensor-core GEMM) ----
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peaks = json.load(open(peaks_path))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        hbm_peak, peak_src = 6800.0, "fallback"
    total_bytes, w_bytes = algorithmic_bytes(s, wl, cyc.ctx)
    R = wl.n_req * wl.L
    gemm_bytes = 0
    gemm_flops = 0
    for _, M, N, K in gemm_shapes(s, wl.n_req * wl.L, R):
        gemm_bytes += 2 * (N * K + M * K) + 4 * M * N
        gemm_flops += 2 * M * N * K
    n_gemm = launches.get("gemm_tc", 1)
    gemm_us = per_cycle.get("gemm_tc", float("nan"))
    tc_peak = float(peaks["bf16_tflops"]) if os.path.exists(peaks_path) else 1900.0
    # the GEMMs' bound: HBM below the ridge (peak flop/s over peak bytes/s), tensor above
    if gemm_flops / gemm_bytes > tc_peak * 1e12 / (hbm_peak * 1e9):
        achieved = (gemm_flops / n_gemm) / (gemm_us / n_gemm * 1e-6) / 1e12
        roofline = {"bound": "tensor", "kernel": "gemm_tc", "achieved": round(achieved, 1),
                    "peak": tc_peak, "peak_source": peak_src, "unit": "TFLOP/s",
                    "frac": round(achieved / tc_peak, 4),
                    "flops_per_launch": int(gemm_flops / n_gemm),
                    "us_per_launch": round(gemm_us / n_gemm, 2), "traffic": None}
    else:
        achieved = (gemm_bytes / n_gemm) / (gemm_us / n_gemm * 1e-6) / 1e9
        roofline = {"bound": "hbm", "kernel": "gemm_tc", "achieved": round(achieved, 1),
                    "peak": hbm_peak, "peak_source": peak_src, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4),
                    "bytes_per_launch": int(gemm_bytes / n_gemm),
                    "us_per_launch": round(gemm_us / n_gemm, 2),
                    "traffic": traffic_from_profile(os.path.join(
                        ROOT, "block_diffusion_speculative_kv_gb300", "csrc", "gemm_tc.cu"))}
    cycle_gbs = total_bytes / (ms_step * 1e-3) / 1e9

    # ---- e2e: C-ABI calls with pinned host buffers, copies in the timed region ----
    h_feats = cyc.feats.cpu().pin_memory()
    h_anchor = cyc.anchor.cpu().pin_memory()
    h_ctx = cyc.ctx_len.cpu().pin_memory()
    outs = [cyc.ids, cyc.lp] + list(cyc.tree)
    h_outs = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = h_feats.numel() * h_feats.element_size() + h_anchor.numel() * 4 + h_ctx.numel() * 4
    d2h = sum(o.numel() * o.element_size() for o in outs)

    def e2e_step():
        cyc.feats.copy_(h_feats, non_blocking=True)
        cyc.anchor.copy_(h_anchor, non_blocking=True)
        cyc.ctx_len.copy_(h_ctx, non_blocking=True)
        cyc.run()
        for h, o in zip(h_outs, outs):
            h.copy_(o, non_blocking=True)

    ms_e2e_total, _ = timed_region(e2e_step, args.steps, 3, world)
    ms_e2e = max_over_ranks(ms_e2e_total / args.steps, world)

    # ---- the other workloads, as sub-records of this line ----
    configs = {}
    if rank == 0 and not args.no_configs and args.workload == 2:
        w = max(args.warmup, 3)
        subs = [("qwen3_8b_b1_t1", lambda: sub_cycle_record(2, args.steps, w, (1.0, 12345), cyc)),
                ("qwen3_4b_b1", lambda: sub_cycle_record(1, args.steps, w)),
                ("qwen3_8b_batch32", lambda: sub_cycle_record(3, max(3, args.steps // 2), w)),
                ("stress", lambda: stress_record(args.steps, w))]
        for name, f in subs:
            try:
                configs[name] = f()
            except Exception as ex:  # report, do not hide
                configs[name] = {"error": f"{type(ex).__name__}: {ex}"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(cyc, args.cpu_budget_s)
        except Exception as ex:  # report, do not hide
            cpu = {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"failed: {type(ex).__name__}: {ex}"}

    value = replica_value(ms_step, world)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4),
        "us_per_cycle": round(ms_step * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "n_layers": s.n_layers, "d": s.d, "heads": [s.n_q, s.n_kv],
                   "head_dim": s.head_dim, "d_ff": s.d_ff, "vocab": s.vocab,
                   "ctx": int(cyc.ctx.max()), "L": wl.L, "K": wl.K, "B": wl.B,
                   "n_req": wl.n_req, "parallelism": "replicas" if world > 1 else "single",
                   "timed": "CUDA graph of the cycle",
                   "l2": "inputs larger than L2 (%.2f GB per cycle vs 129 MB)" % (total_bytes / 1e9)},
        "roofline": roofline,
        "cycle_hbm": {"algorithmic_bytes": int(total_bytes), "achieved_gbs": round(cycle_gbs, 1),
                      "frac": round(cycle_gbs / hbm_peak, 4)},
        "kernel_us_per_cycle": {k: round(v, 1) for k, v in per_cycle.items()},
        "kernel_share": shares,
        "accept_us": round(accept_us, 2),
        "us_per_cycle_with_accept": round(ms_step * 1e3 + accept_us, 1),
        "e2e": {"value": round(replica_value(ms_e2e, world), 2), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(ms_e2e, 4), "path": "C-ABI calls, eager"},
        "gpu_launches": launches_per_cycle * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
