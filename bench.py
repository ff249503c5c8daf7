"""Benchmark of one tree speculative decoding verify step on GB300.

A step is one pass of the whole hot path over one batch of seeded synthetic
input: jt_tree_build (top-W per depth + best-first expansion), then
jt_tree_attn_paged (tree-causal attention over the paged bf16 KV cache, fed
by the build's ancestor sets), then jt_verify_accept with the greedy rule
and with the margin rule (t = 0.8).  Metric: tree-node tokens per second.

Default workload (--config 4): the KV-bandwidth-bound high-load case of a
Qwen3-8B-shaped attention layer (32 query / 8 KV heads, head dim 128, bf16):
32 sequences of prefix 32768, tree budget 64 (N=8, W=4), vocab 151936, pages
randomly permuted in the pool (4.3 GB of K/V, far larger than L2).  The
other workloads (--config 2: batch 1, prefix 4096, budget 256; 3: a ragged
serving batch; 5: the full verify step of 8 sequences) run with --config.

`value` is the whole verify step's rate (tree-node tokens per second of the
step: build + attention + both acceptance rules); the attention call's own
rate is `roofline.attn_tokens_per_s`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

Rank 0 prints one JSON line.  With torchrun (N > 1) every rank runs an
independent replica on its own GPU (the path has no cross-GPU exchange).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tree_speculative_decoding_jt_gb300 import workloads as wk  # noqa: E402

METRIC = "tree-verify attention tree-node-tokens/sec and % of roofline (HBM GB/s) at 1 GB300"
UNIT = "tree-node tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------
# Multi-rank host logic (N > 1): every rank runs an independent replica on
# its own GPU and its own seeded batch; the job's time is the slowest rank's.
# --------------------------------------------------------------------------
def replica_seed(config: int, rank: int) -> int:
    """Seed of rank `rank`'s batch: the workload's default seed for rank 0,
    distinct seeds for the other replicas."""
    return 1000 + config + 7919 * rank


def max_over_ranks(values, device, world):
    """Element-wise maximum of a list of floats over all ranks (identity at
    world == 1)."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(units_per_rank: int, seconds: float, world: int) -> float:
    """Units all ranks processed per second of the slowest rank's time."""
    return world * units_per_rank / seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def attn_algorithmic(wl, depth):
    """Algorithmic bytes and FLOPs of one attention call: K and V of the
    prefix + tree slots once, q and o once; 4*D flops per (query head,
    visible key) for QK^T and PV, visible keys = prefix + ancestors."""
    c = wl.cfg
    Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
    esz = 2 if c["dtype"] == "bf16" else 4
    B = np.diff(wl.tree_off)
    slots = int(np.sum(wl.prefix_len.astype(np.int64) + B))
    kv_bytes = slots * Hkv * D * 2 * esz
    qo_bytes = 2 * wl.total * Hq * D * esz
    flops = 0
    for b in range(wl.nseq):
        o, e = int(wl.tree_off[b]), int(wl.tree_off[b + 1])
        flops += int(np.sum(int(wl.prefix_len[b]) + depth[o:e].astype(np.int64) + 1)) * 4 * Hq * D
    return kv_bytes + qo_bytes, flops


class ClockSampler:
    """nvidia-smi clock/throttle samples around the timed region.

    start() launches `nvidia-smi -lms PERIOD` and returns once its first
    sample has arrived (so sampling is live before the region starts);
    mark_start()/mark_end() bracket the timed region; stop() waits for one
    more sample after the region, then ends the process and joins the
    reader.  summary() reports the samples that fall inside the region,
    widened by one period on each side (a region shorter than a period still
    gets its nearest samples under load), beside the total count."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.thread = None
        self.lines = []   # (host time, csv line)
        self.t_start = self.t_end = None

    def start(self, wait_s=10.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.monotonic()
        while not self.lines and time.monotonic() - t0 < wait_s and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def stop(self, wait_s=3.0):
        if self.proc is None:
            return
        t0 = time.monotonic()
        end = self.t_end if self.t_end is not None else t0
        while (not self.lines or self.lines[-1][0] <= end) and time.monotonic() - t0 < wait_s \
                and self.proc.poll() is None:
            time.sleep(0.01)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        pad = self.PERIOD_MS / 1000.0
        t0 = (self.t_start or 0.0) - pad
        t1 = (self.t_end or float("inf")) + pad
        sm, mx, reasons, n_all = [], [], set(), 0
        for t, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                a, b = float(f[1]), float(f[2])
            except ValueError:
                continue
            n_all += 1
            if not t0 <= t <= t1:
                continue
            sm.append(a)
            mx.append(b)
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": sorted(reasons), "samples": len(sm), "samples_total": n_all,
               "window": f"timed region +/- {self.PERIOD_MS} ms (nvidia-smi -lms {self.PERIOD_MS})"}
        if not sm:
            out["note"] = "no sample fell in the window"
        return out


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_file, workload, kernel=None):
    """DRAM bytes of one main attention-kernel launch on `workload` from the
    committed ncu summaries (profiles/traffic.json, one entry per workload
    and kernel), or None when there is no capture for this workload and
    kernel or it was taken on a different version of the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        h = source_hash([kernel_file])
        for e in d.get("entries", []):
            if (e.get("workload") == workload and e.get("source_hash") == h
                    and (kernel is None or e.get("kernel") == kernel)):
                return e.get("dram_bytes_per_launch")
        return None
    except (ValueError, OSError):
        return None


# --------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# --------------------------------------------------------------------------
def held_policy(budgets, N, W):
    """Adaptive-policy parameters that hold every request's budget: every
    request is confident (log_conf = -inf) and none is accepting
    (acc_thresh = +inf), so B never moves; width W, depth N.  The emitted
    trees are then the fixed workload's, and the step measures the policy's
    own cost in the loop."""
    return dict(b_min=int(min(budgets)), b_max=int(max(budgets)), node_cap=0, w_min=W, n_min=N, n_slack=N,
                beta=0.25, log_conf=-math.inf, acc_thresh=math.inf)


def oracle_build(wl, alpha, adaptive=False):
    """The oracle's tree build of the step: plain, entropy-mixed scores, or
    the adaptive policy (held budgets) followed by the capped expansion."""
    import oracle

    c = wl.cfg
    if adaptive:
        tb = oracle.tree_build(wl.draft_logits, wl.root_token,
                               np.arange(wl.nseq + 1, dtype=np.int32), c["W"])
        budgets = np.diff(wl.tree_off)
        pol = oracle.tree_policy(tb["lp"], None, budgets, np.zeros(wl.nseq), **held_policy(budgets, c["N"], c["W"]))
        return oracle.tree_expand_capped(tb["tok"], tb["lp"], wl.root_token, pol["tree_off"], c["N"], c["W"],
                                         w_cap=pol["w_cap"], n_cap=pol["n_cap"])
    if alpha == 0.0:
        return oracle.tree_build(wl.draft_logits, wl.root_token, wl.tree_off, c["W"])
    return oracle.tree_build_mixed(wl.draft_logits, wl.root_token, wl.tree_off, c["W"], alpha)


def oracle_accept(wl, target, parent, token, uniforms):
    """The oracle's acceptance rules of the step (greedy, margin, and the
    temperature-1 rule when uniforms are given)."""
    import oracle

    c = wl.cfg
    oracle.verify_accept(target, parent, token, wl.tree_off, c["N"], 0)
    oracle.verify_accept(target, parent, token, wl.tree_off, c["N"], 1, math.log(c["t"]))
    if uniforms is not None:
        oracle.verify_accept_stochastic(target, wl.draft_logits, parent, token, wl.tree_off, c["N"],
                                        uniforms[0], uniforms[1])


def step_uniforms(cfg, rank, total):
    """Seeded uniforms of the temperature-1 acceptance, one pair per node."""
    u = np.random.default_rng(replica_seed(cfg, rank) + 1).random((2, total))
    return u[0].copy(), u[1].copy()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_sample(wl, attn_k, alpha, uniforms, adaptive, threads=1, target_s=6.0):
    """The oracle, as it stands, on a bounded sample: the whole build and the
    acceptance rules of the batch (single calls) and the attention of attn_k
    nodes spread over the batch (attn_k = 0: as many as about target_s
    seconds of one thread's work, from the time of two nodes); with threads
    > 1 the attention runs on `threads` host threads, each over a disjoint
    node set of that size (the C oracle runs outside the interpreter lock),
    and the attention cost per node is the wall time over all of them.
    Returns (tree-node tokens/s, seconds of oracle work, nodes per thread)."""
    import concurrent.futures
    import oracle

    t0 = time.perf_counter()
    tr = oracle_build(wl, alpha, adaptive)
    t1 = time.perf_counter()
    # every input of the timed oracle calls comes from the oracle's own tree
    target = wk.target_logits(wl, tr["parent"], tr["token"])

    def attn(rows):
        oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len, wl.tree_off,
                         tr["parent"], wl.scale, rows=rows)

    if attn_k <= 0:
        tc = time.perf_counter()
        attn(attn_sample_nodes(wl, 2))
        per = (time.perf_counter() - tc) / 2
        attn_k = int(max(4, min(512, target_s / max(per, 1e-6))))
    attn_nodes = attn_sample_nodes(wl, attn_k)
    t1b = time.perf_counter()
    if threads <= 1:
        attn(attn_nodes)
        n_attn = len(attn_nodes)
    else:
        k = len(attn_nodes)
        sets = [((attn_nodes + i * 7919) % wl.total).astype(np.int32) for i in range(threads)]
        with concurrent.futures.ThreadPoolExecutor(threads) as ex:
            list(ex.map(attn, sets))
        n_attn = k * threads
    t2 = time.perf_counter()
    oracle_accept(wl, target, tr["parent"], tr["token"], uniforms)
    t3 = time.perf_counter()
    # per-node cost of the whole step: build and accept per node of the
    # batch, attention per sampled node
    per_node = (t1 - t0) / wl.total + (t2 - t1b) / n_attn + (t3 - t2) / wl.total
    return 1.0 / per_node, (t1 - t0) + (t3 - t1b), len(attn_nodes)


def attn_sample_nodes(wl, k):
    step = max(1, wl.total // k)
    return np.arange(0, wl.total, step, dtype=np.int32)[:k]


def step_name(args):
    build = "tree_build" if args.alpha == 0.0 else f"tree_build_mixed(alpha={args.alpha:g})"
    if args.adaptive:
        build = "tree_build_adaptive(policy fed the last greedy accept_len, holding each budget)"
    return (build + " + tree_attn_paged + verify_accept(greedy) + verify_accept(margin t=0.8)"
            + (" + verify_accept_stochastic(T=1)" if args.stochastic else ""))


def make_workload(args, seed):
    """The seeded workload of --config; --nseq keeps only its first
    sequences (a reduced shape for profiler captures, named as such)."""
    if not args.nseq:
        return wk.make(args.config, seed=seed)
    c = wk.CONFIGS[args.config]
    if not 1 <= args.nseq <= c["nseq"]:
        raise SystemExit(f"--nseq must lie in [1, {c['nseq']}]")
    budgets = c["budgets"] if len(c["budgets"]) == 1 else c["budgets"][:args.nseq]
    name = f"{c['name']} (first {args.nseq} of {c['nseq']} sequences)"
    return wk.make(args.config, seed=seed, overrides={"nseq": args.nseq, "budgets": budgets, "name": name})


def attn_kernel(D, Hq, Hkv, max_tree):
    """The attention kernel the library picks (its rule, mirrored): for head
    dim 128 the CTA-pair kernel when every (sequence, KV head) has one
    query-tile pair at max_tree, else the single-SM kernel; JT_ATTN_KERNEL
    = pair / single overrides; head dim 64 always runs the single-SM one."""
    if D != 128:
        return "single"
    env = os.environ.get("JT_ATTN_KERNEL")
    if env in ("pair", "single"):
        return env
    npt = 128 // (Hq // Hkv)
    npairs = (-(-max_tree // npt) + 1) // 2
    return "pair" if npairs == 1 else "single"


def attn_split_mode(nseq, Hq, Hkv, max_tree, max_pages, slots):
    """Whether jt_tree_attn_paged runs in split mode (a second, combine
    kernel): the library's rule -- at most half as many (sequence, KV head,
    query-tile pair) units as work slots (one per SM, or one per resident CTA
    pair: SMs / 2), and at least two key splits each."""
    npt = 128 // (Hq // Hkv)
    units = nseq * Hkv * ((-(-max_tree // npt) + 1) // 2)
    tmax = -(-max_pages * 16 // 128)
    if units <= 0 or 2 * units > slots:
        return False
    return min(slots // units, max(1, tmax // 2), 32) >= 2


def config_dict(args, wl, world):
    """The workload description both arms print (identical dicts for the
    same command line)."""
    c = wl.cfg
    return {"workload": c["name"], "nseq": wl.nseq, "tree_nodes": wl.total,
            "prefix_len": [int(x) for x in wl.prefix_len[:4]] + (["..."] if wl.nseq > 4 else []),
            "Hq": c["Hq"], "Hkv": c["Hkv"], "head_dim": c["D"], "N": c["N"], "W": c["W"], "V": c["V"],
            "step": step_name(args),
            "l2": f"flushed before every step ({args.flush_mb} MiB write)",
            "parallelism": f"replicas x{world}"}


VALUE_IS = ("whole verify step: tree-node tokens per second of build + attention + acceptance "
            "(attention alone: roofline.attn_tokens_per_s)")


def run_reference(args, rank):
    """The oracle, as it stands, on the host cores.  One reference step is
    the attention of one tree node per host thread, run concurrently
    (rotating over the batch; the C oracle runs outside the interpreter
    lock), plus the matching share of the full tree build and of the
    acceptance rules, which are timed once over the whole batch; a run of K
    steps costs about K single-node attention times and stays within
    minutes."""
    if rank != 0:
        return
    import concurrent.futures
    import oracle

    wl = make_workload(args, replica_seed(args.config, 0))
    c = wl.cfg
    t0 = time.perf_counter()
    tr = oracle_build(wl, args.alpha, args.adaptive)
    t_build = time.perf_counter() - t0
    target = wk.target_logits(wl, tr["parent"], tr["token"])
    uniforms = step_uniforms(args.config, 0, wl.total) if args.stochastic else None
    t0 = time.perf_counter()
    oracle_accept(wl, target, tr["parent"], tr["token"], uniforms)
    t_accept = time.perf_counter() - t0

    def attn_one(n):
        oracle.tree_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.prefix_len, wl.tree_off,
                         tr["parent"], wl.scale, rows=np.array([n], np.int32))

    threads = min(host_cores(), 64)
    pool = concurrent.futures.ThreadPoolExecutor(threads)
    for i in range(min(args.warmup, 3)):
        list(pool.map(attn_one, [(i * threads + t) % wl.total for t in range(threads)]))
    # K steps, or as many as fit in the time budget (a long-prefix node costs
    # a fraction of a second of fp64 work per thread)
    times = []
    t_start = time.perf_counter()
    for i in range(args.steps):
        t0 = time.perf_counter()
        list(pool.map(attn_one, [((i * threads + t) * 37) % wl.total for t in range(threads)]))
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > args.ref_budget_s:
            break
    wall = time.perf_counter() - t_start
    pool.shutdown()
    per_node = t_build / wl.total + t_accept / wl.total + statistics.mean(times) / threads
    value = 1.0 / per_node
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_node,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "value_is": VALUE_IS, "config": config_dict(args, wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"tree build ({t_build:.2f} s) and the acceptance rules "
                                   f"({t_accept:.2f} s) over all {wl.total} nodes once (one thread), "
                                   f"attention of {threads} nodes per step on {threads} host threads "
                                   f"for {len(times)} of {args.steps} steps ({wall:.1f} s, budget "
                                   f"{args.ref_budget_s:g} s); C, fp64"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--nseq", type=int, default=0,
                    help="keep only the first NSEQ sequences of the workload (reduced shapes for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-attn-nodes", type=int, default=0,
                    help="attention nodes per host thread in the CPU baseline (0: sized to the prefix)")
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="--impl reference: stop after the step that crosses this many seconds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--no-graph", action="store_true", help="launch every call eagerly")
    ap.add_argument("--stochastic", action="store_true",
                    help="add the temperature-1 acceptance (jt_verify_accept_stochastic) to the step")
    ap.add_argument("--alpha", type=float, default=0.0,
                    help="entropy weight of the tree build's step scores (jt_tree_build_mixed); 0 = plain")
    ap.add_argument("--adaptive", action="store_true",
                    help="build through jt_tree_build_adaptive (top-W, policy, capped expansion), the "
                         "policy fed each step's greedy accept_len and holding every budget")
    ap.add_argument("--serial", action="store_true",
                    help="one stream: attention, then the acceptance rules (default: acceptance on side "
                         "streams beside the attention)")
    args = ap.parse_args()
    if not 0.0 <= args.alpha <= 1.0:
        raise SystemExit("--alpha must lie in [0, 1]")
    if args.adaptive and args.alpha > 0:
        raise SystemExit("--adaptive and --alpha do not combine")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    import tree_speculative_decoding_jt_gb300 as jt

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if world > 1:
            dist.barrier()

    cfg = args.config
    wl = make_workload(args, replica_seed(cfg, rank))
    c = wl.cfg
    dev = torch.device("cuda", local_rank)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    h = {  # host copies (pinned) of every per-step input, for the end-to-end leg
        "draft": torch.from_numpy(wl.draft_logits),
        "root": torch.from_numpy(wl.root_token),
        "off": torch.from_numpy(wl.tree_off),
        "plen": torch.from_numpy(wl.prefix_len),
        "bt": torch.from_numpy(wl.block_table),
        "q": torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16) if wl.q.dtype == np.uint16 else torch.from_numpy(wl.q),
        "k": torch.from_numpy(wl.k_cache.view(np.int16)).view(torch.bfloat16) if wl.k_cache.dtype == np.uint16 else torch.from_numpy(wl.k_cache),
        "v": torch.from_numpy(wl.v_cache.view(np.int16)).view(torch.bfloat16) if wl.v_cache.dtype == np.uint16 else torch.from_numpy(wl.v_cache),
    }
    d = {k: v.to(dev) for k, v in h.items()}
    total, nseq, N, W = wl.total, wl.nseq, c["N"], c["W"]
    max_tree = int(np.diff(wl.tree_off).max())
    Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
    max_pages = wl.block_table.shape[1]
    log_t = math.log(c["t"])

    # outputs and workspaces, allocated once (node arrays sized to the
    # policy's capacity in adaptive mode)
    budgets = np.diff(wl.tree_off)
    cap = nseq * int(budgets.max()) if args.adaptive else total
    parent = torch.empty(cap, dtype=torch.int32, device=dev)
    token = torch.empty_like(parent)
    depth = torch.empty_like(parent)
    anc = torch.empty((cap, 8), dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty((total, Hq), dtype=torch.float32, device=dev)
    acc = [torch.full((nseq,), -1, dtype=torch.int32, device=dev) for _ in range(3)]
    path = [torch.empty((nseq, N + 1), dtype=torch.int32, device=dev) for _ in range(3)]
    bonus = [torch.empty(nseq, dtype=torch.int32, device=dev) for _ in range(3)]
    build_op = jt.JT_OP_TREE_BUILD_MIXED if args.alpha > 0 else jt.JT_OP_TREE_BUILD
    ws_b = jt.workspace(jt.jt_workspace_size(build_op, nseq, N, W, c["V"]), dev)

    if args.adaptive:
        prm = jt.policy_params(**held_policy(budgets, N, W))
        pol_state = (to_dev(budgets.astype(np.int32)), torch.zeros(nseq, dtype=torch.float64, device=dev))
        pol_out = (torch.empty(nseq + 1, dtype=torch.int32, device=dev),
                   torch.empty(nseq, dtype=torch.int32, device=dev), torch.empty(nseq, dtype=torch.int32, device=dev))

    def offs(inp):
        return pol_out[0] if args.adaptive else inp["off"]

    def build(inp):
        if args.adaptive:   # acc[0]: the previous step's greedy accepted lengths
            jt.jt_tree_build_adaptive(inp["draft"], inp["root"], acc[0], pol_state[0], pol_state[1], W, prm,
                                      capacity=cap, out=pol_out + (parent, token, depth, anc), ws=ws_b)
        elif args.alpha > 0:
            jt.jt_tree_build_mixed(inp["draft"], inp["root"], inp["off"], W, args.alpha, total_nodes=total,
                                   out=(parent, token, depth, anc), ws=ws_b)
        else:
            jt.jt_tree_build(inp["draft"], inp["root"], inp["off"], W, total_nodes=total,
                             out=(parent, token, depth, anc), ws=ws_b)
    ws_a = jt.workspace(jt.jt_workspace_size(jt.JT_OP_TREE_ATTN, nseq, 0, 0, 0, total, Hq, Hkv, D,
                                             max_pages, max_tree), dev)
    ws_v = [jt.workspace(jt.jt_workspace_size(jt.JT_OP_VERIFY_ACCEPT, nseq, 0, 0, 0, total), dev)
            for _ in range(3)]

    # target logits need the drafted tokens: build the tree once, then draw
    build(d)
    jt.jt_check(ws_b)
    if args.adaptive:   # the held policy must reproduce the workload's offsets
        assert np.array_equal(pol_out[0].cpu().numpy(), wl.tree_off), "adaptive policy moved a budget"
    par_h, tok_h, dep_h = (t.cpu().numpy()[:total] for t in (parent, token, depth))
    target_np = wk.target_logits(wl, par_h, tok_h)
    h["target"] = torch.from_numpy(target_np)
    d["target"] = h["target"].to(dev)
    uniforms = step_uniforms(cfg, rank, total) if args.stochastic else None
    if uniforms is not None:
        h["u_acc"], h["u_bon"] = torch.from_numpy(uniforms[0]), torch.from_numpy(uniforms[1])
        d["u_acc"], d["u_bon"] = h["u_acc"].to(dev), h["u_bon"].to(dev)

    stream = torch.cuda.current_stream()
    attn_ev = []
    # The acceptance rules read the tree and the target logits, not the
    # attention output: after the build they run on side streams beside the
    # attention (joined before the step ends), unless --serial.
    side = [torch.cuda.Stream(device=dev) for _ in range(3)]

    def accepts(inp, i):
        if i < 2:
            jt.jt_verify_accept(inp["target"], parent, token, offs(inp), N,
                                rule=(jt.JT_RULE_GREEDY, jt.JT_RULE_MARGIN)[i], log_t=log_t,
                                out=(acc[i], path[i], bonus[i]), ws=ws_v[i])
        else:
            jt.jt_verify_accept_stochastic(inp["target"], inp["draft"], parent, token, offs(inp), N,
                                           inp["u_acc"], inp["u_bon"], out=(acc[2], path[2], bonus[2]),
                                           ws=ws_v[2])

    n_acc = 3 if args.stochastic else 2

    def attention(inp):
        jt.jt_tree_attn_paged(inp["q"], inp["k"], inp["v"], inp["bt"], inp["plen"], offs(inp), anc,
                              scale=wl.scale, max_tree=max_tree, out=out, lse=lse, ws=ws_a)

    def step(inp):
        build(inp)
        if args.serial:
            attention(inp)
            for i in range(n_acc):
                accepts(inp, i)
            return
        # acceptance first: its cluster kernels then find free SMs before the
        # attention fills the GPU (the other order measured 83.7 vs 80.6 us)
        main = torch.cuda.current_stream()
        built = torch.cuda.Event()
        built.record(main)
        for i in range(n_acc):
            side[i].wait_event(built)
            with torch.cuda.stream(side[i]):
                accepts(inp, i)
        attention(inp)
        for i in range(n_acc):
            main.wait_stream(side[i])

    flush = torch.empty(args.flush_mb * (1 << 20), dtype=torch.uint8, device=dev)
    # clock sampling is live from the warm-up on, so the GPU is under load
    # when the timed region starts
    clocks = ClockSampler(local_rank).start()
    for _ in range(args.warmup):
        flush.zero_()
        step(d)
    torch.cuda.synchronize()
    for ws in (ws_b, ws_a, *ws_v):
        jt.jt_check(ws)

    def attn_only(inp):
        jt.jt_tree_attn_paged(inp["q"], inp["k"], inp["v"], inp["bt"], inp["plen"], offs(inp), anc,
                              scale=wl.scale, max_tree=max_tree, out=out, lse=lse, ws=ws_a)

    # The step's kernels are replayed from a CUDA graph (as a serving engine
    # would), so host launch overhead stays out of the device timeline.
    g_step, g_attn = None, None
    if not args.no_graph:
        g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            step(d)
        with torch.cuda.graph(g_attn):
            attn_only(d)
        for _ in range(args.warmup):
            flush.zero_()
            g_step.replay()
        torch.cuda.synchronize()
        for ws in (ws_b, ws_a, *ws_v):
            jt.jt_check(ws)

    # ---- timed region (inputs resident in HBM; L2 flushed before each step)
    evs = []
    barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if g_step is not None:
            g_step.replay()
        else:
            step(d)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t_wall0
    clocks.mark_end()
    clocks.stop()
    # the dominant kernel alone, same inputs, same L2 flush, for the roofline
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if g_attn is not None:
            g_attn.replay()
        else:
            attn_only(d)
        e1.record(stream)
        attn_ev.append((e0, e1))
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    ms = statistics.mean(step_ms)
    ms_median = statistics.median(step_ms)
    attn_mean = statistics.mean(attn_ms)
    attn_median = statistics.median(attn_ms)
    ms, attn_mean = max_over_ranks([ms, attn_mean], dev, world)
    value = whole_job_rate(total, ms * 1e-3, world)

    # ---- end to end: pinned host inputs -> C-ABI calls -> host results
    e2e = None
    if args.e2e_steps > 0:
        hp = {k: v.pin_memory() for k, v in h.items()}
        results = [parent, token, out, acc[0], path[0], bonus[0], acc[1], path[1], bonus[1]]
        if args.stochastic:
            results += [acc[2], path[2], bonus[2]]
        res_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in results]
        h2d = sum(v.numel() * v.element_size() for v in hp.values())
        d2h = sum(v.numel() * v.element_size() for v in res_h)
        dd = {k: torch.empty_like(v) for k, v in d.items()}
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            for k in hp:
                dd[k].copy_(hp[k], non_blocking=True)
            step(dd)
            for dst, src in zip(res_h, results):
                dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize()
        e2e_s = (time.perf_counter() - t0) / args.e2e_steps
        e2e_s = max_over_ranks([e2e_s], dev, world)[0]
        e2e = {"value": whole_job_rate(total, e2e_s, world), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps,
               "h2d_gbs": h2d / e2e_s / 1e9}

    # ---- roofline of the dominant kernel (the attention call)
    peaks, peak_src = load_peaks()
    bytes_a, flops_a = attn_algorithmic(wl, dep_h)
    t_hbm = bytes_a / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops_a / (peaks["bf16_tflops"] * 1e12)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": flops_a / (attn_mean * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": bytes_a / (attn_mean * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    kern = attn_kernel(c["D"], c["Hq"], c["Hkv"], max_tree)
    kname = "tree_attn_pair_kernel" if kern == "pair" else f"tree_attn_tc_kernel<{c['D']}>"
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    split = attn_split_mode(nseq, Hq, Hkv, max_tree, max_pages, sms // 2 if kern == "pair" else sms)
    roof["traffic"] = profiled_traffic("tree_speculative_decoding_jt_gb300/csrc/tree_attn.cu", c["name"], kname)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback"
    roof["kernel"] = f"jt_tree_attn_paged ({kname}" + (" + tree_attn_combine_kernel, split mode)" if split else ")")
    roof["algorithmic_bytes"] = int(bytes_a)
    roof["algorithmic_flops"] = int(flops_a)
    roof["attn_ms"] = attn_mean
    roof["attn_ms_median"] = attn_median
    roof["attn_tokens_per_s"] = total / (attn_mean * 1e-3)
    # the same achieved rate against the other denominators: the sustained
    # measured bf16 rate (a long GEMM loop under the power cap) and the
    # nominal figures (2.25 PFLOP/s dense bf16, 7.9 TB/s HBM3e)
    if roof["bound"] == "tensor":
        roof["frac_of_sustained"] = roof["achieved"] / peaks.get("bf16_tflops_sustained", roof["peak"])
        roof["frac_of_nominal"] = roof["achieved"] / 2250.0
    else:
        roof["frac_of_nominal"] = roof["achieved"] / 7900.0

    # ---- CPU baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v1, secs1, k1 = cpu_oracle_sample(wl, args.cpu_attn_nodes, args.alpha, uniforms, args.adaptive)
        cores = min(host_cores(), 64)
        vn, secsn, kn = cpu_oracle_sample(wl, k1, args.alpha, uniforms, args.adaptive, threads=cores)
        cpu = {"value": vn, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"full tree build and the step's acceptance rules over all {total} nodes "
                         f"(one thread), attention for {kn} nodes on each of {cores} host threads "
                         f"({secsn:.1f} s; C, fp64)",
               "single_thread": {"value": v1, "cores": 1,
                                 "sample": f"same, attention for {k1} of {total} nodes on one thread "
                                           f"({secs1:.1f} s)"}}

    # our kernels per step: the build (top-W partials, then the expansion
    # with the row merge; the adaptive build: partials, row merge, policy,
    # capped expansion), the attention (one kernel; plus the combine in
    # split mode), the acceptance rules
    launches_per_step = ((4 if args.adaptive else 2) + (2 if split else 1) + 2 + (1 if args.stochastic else 0))
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_median, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "value_is": VALUE_IS, "config": config_dict(args, wl, world),
            "schedule": ("one stream" if args.serial else
                         "acceptance on side streams beside the attention (after the build)"),
            "launch": "eager" if args.no_graph else "cuda_graph replay of the step",
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
