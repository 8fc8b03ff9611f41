#!/usr/bin/env python3
"""Spec-tree step benchmark: steps/s of topk + tree build + tree attention +
acceptance on one GB300 (or N replicas, one per GPU), printed as one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Timed region: exactly K steps of the four library calls, replayed from CUDA
graphs (one step per input set in turn), rotating over enough input sets that
their total exceeds twice the 129 MB L2 (so every step reads its inputs from
HBM), bracketed by a barrier and device syncs, timed with CUDA events on the
launching stream; max over ranks.  Per-kernel durations for the roofline come
from a second pass: each stage launched back to back over the input sets
between two events, queued behind a GPU sleep so host launch gaps do not count.
The line also carries the same steps launched eagerly (no graph, the host's
launch cost included) and the step's roofline: the per-stage minimum times at
the measured peaks, summed, over the measured step time.
With N > 1 (torchrun) every rank is an independent replica on its own inputs.
"""
import os

# the oracle baseline runs single-threaded; pin BLAS before numpy loads
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
DEFAULT_WORKLOAD = "long_ctx_b4"

# DRAM bytes (read + write) of one launch (ncu dram__bytes_read.sum +
# dram__bytes_write.sum, one capture of the workload); an entry counts only
# while the kernel's sources still hash to `src`
KNOWN_TRAFFIC = {
    ("topk_softmax", "long_ctx_b4"): {"bytes": 19487488, "src": "b3ccdb7b481d15a2"},
    ("tree_attn", "long_ctx_b4"): {"bytes": 548102144, "src": "abb308e9ee576ad9"},
    ("accept", "long_ctx_b4"): {"bytes": 159599872, "src": "46cf3ac181492cfd"},
    ("tree_attn", "llama31_8b_b16_paged"): {"bytes": 295353856, "src": "abb308e9ee576ad9"},
    ("accept", "llama31_8b_b16_paged"): {"bytes": 50337024, "src": "46cf3ac181492cfd"},
    ("topk_softmax", "qwen3_8b_b1"): {"bytes": 4905216, "src": "b3ccdb7b481d15a2"},
    ("tree_build", "qwen3_8b_b1"): {"bytes": 29440, "src": "48ae66f3c4acd9a7"},
    ("tree_attn", "qwen3_8b_b1"): {"bytes": 17634048, "src": "abb308e9ee576ad9"},
    ("accept", "qwen3_8b_b1"): {"bytes": 19477760, "src": "46cf3ac181492cfd"},
    ("tree_build", "long_ctx_b4"): {"bytes": 34048, "src": "48ae66f3c4acd9a7"},
}
KERNEL_SOURCES = {
    "topk_softmax": ("topk_softmax.cu", "sm100_ptx.cuh", "common.cuh"),
    "tree_build": ("tree_build.cu", "common.cuh"),
    "tree_attn": ("tree_attn.cu", "sm100_ptx.cuh", "common.cuh"),
    "accept": ("accept.cu", "sm100_ptx.cuh", "common.cuh"),
}


def kernel_source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "tree_speculative_decoding_bastion_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def known_traffic(kernel, workload):
    t = KNOWN_TRAFFIC.get((kernel, workload))
    if t and t["src"] == kernel_source_hash(kernel):
        return t["bytes"]
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------


# ----------------------------------------------------------------------------
# replicas: one process per GPU, each on its own inputs (weak scaling)
# ----------------------------------------------------------------------------


def replica_seed(rank, r):
    """Seed of input set r on replica `rank`: every replica draws its own batch."""
    return 1000 * rank + r


def max_over_ranks(x, world):
    """The largest of the ranks' values (the job's time is its slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, steps, ms):
    """Whole-job steps/s: every rank ran `steps` steps in at most `ms`."""
    return world * steps / (ms / 1e3)


# What the oracle pool's workers read.  Filled in the parent before the pool
# forks (no GPU call has been made by then), so the workers inherit it.
_ORACLE = {}


def host_cores():
    """Cores this process may run on (the affinity mask, else the CPU count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


class _F32View:
    """float32 values of a stored (bf16 bits or float32) array, converted on indexing."""

    def __init__(self, a, dtype):
        self.a, self.dtype, self.shape = a, dtype, a.shape

    def __getitem__(self, idx):
        return I.as_f32(self.a[idx], self.dtype)


def _w_topk(r0, r1):
    import oracle
    o = _ORACLE
    wl = o["wl"]
    t = time.perf_counter()
    x = I.as_f32(o["inp"].logits.reshape(wl.B * wl.K, wl.V)[r0:r1], wl.dtype)
    oracle.topk_softmax(x, wl.topk)
    return time.perf_counter() - t


def _w_tree(b):
    import oracle
    o = _ORACLE
    wl, inp, s1 = o["wl"], o["inp"], o["s1"]
    t = time.perf_counter()
    oracle.tree_build(s1["ids"][b:b + 1], s1["lg"][b:b + 1], s1["lse"][b:b + 1], inp.root_tok[b:b + 1],
                      inp.ctx_len[b:b + 1], wl.n_min, wl.n_max, inp.C, inp.L_AR)
    return time.perf_counter() - t


def _w_attn(rows):
    import oracle
    o = _ORACLE
    wl, inp, T = o["wl"], o["inp"], o["tree"]
    v = lambda a: _F32View(a, wl.dtype)
    t = time.perf_counter()
    oracle.tree_attention(v(inp.q), v(inp.k_tree), v(inp.v_tree), v(inp.k_ctx), v(inp.v_ctx), inp.ctx_len,
                          T["parent"], T["n"], wl.Hkv, inp.scale, block_table=inp.block_table,
                          page_size=wl.page_size, rows=rows)
    return time.perf_counter() - t


def _w_accept(b):
    import oracle
    o = _ORACLE
    wl, T = o["wl"], o["tree"]
    t = time.perf_counter()
    oracle.accept(_F32View(o["target"][b:b + 1], wl.dtype), T["n"][b:b + 1], T["parent"][b:b + 1],
                  T["token"][b:b + 1], wl.K)
    return time.perf_counter() - t


class OracleBench:
    """The CPU oracle (``oracle/``, numpy float64, as it stands) timed on the
    host cores over one step of the workload.

    A step runs stages 1, 2 and 4 whole (every drafter row, every request's
    tree, every tree node's argmax and walk) and stage 3 on a sample: ROWS
    (node, head) rows from each of up to P (request, KV head) groups, drawn
    afresh every step.  Attention rows are independent and equally costly
    within a group, so the step's full time is modelled as the measured wall
    time of stages 1, 2 and 4 plus the sampled attention's CPU seconds scaled
    to every row of the batch and spread evenly over the P cores.  The work is
    spread over P worker processes forked before any GPU call (one BLAS thread
    each); P = 1 runs it in this process.
    """

    ROWS = 16

    def __init__(self, wl, inp):
        import oracle
        self.wl, self.inp = wl, inp
        # untimed pre-pass: the oracle's own tree and the target logits for it
        x = I.as_f32(inp.logits, wl.dtype).reshape(wl.B * wl.K, wl.V)
        ids, lg, q, lse = oracle.topk_softmax(x, wl.topk)
        s1 = {"ids": ids.reshape(wl.B, wl.K, -1), "lg": lg.reshape(wl.B, wl.K, -1), "lse": lse.reshape(wl.B, wl.K)}
        T = oracle.stack_trees(oracle.tree_build(s1["ids"], s1["lg"], s1["lse"], inp.root_tok, inp.ctx_len,
                                                 wl.n_min, wl.n_max, inp.C, inp.L_AR))
        target = I.make_target_logits(inp, T["depth"], T["n"])
        _ORACLE.update(wl=wl, inp=inp, s1=s1, tree=T, target=target)
        self.T = T
        self.total_rows = int(sum(int(T["n"][b]) for b in range(wl.B))) * wl.Hq
        self.groups = [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hkv)]
        self.pool = None
        self.P = 1
        self.count = 0

    def start_pool(self, P):
        import multiprocessing as mp
        self.P = max(1, int(P))
        if self.P > 1:
            self.pool = mp.get_context("fork").Pool(self.P)

    def close(self):
        if self.pool is not None:
            self.pool.terminate()
            self.pool.join()
            self.pool = None

    def _sample_rows(self):
        wl, T = self.wl, self.T
        rng = np.random.default_rng(self.count)
        self.count += 1
        pick = rng.choice(len(self.groups), size=min(self.P, len(self.groups)), replace=False)
        tasks = []
        for j in sorted(pick):
            b, kvh = self.groups[j]
            nb = int(T["n"][b])
            cand = [(b, i, kvh * wl.g + h) for i in range(nb) for h in range(wl.g)]
            sel = rng.choice(len(cand), size=min(self.ROWS, len(cand)), replace=False)
            tasks.append([cand[k] for k in sorted(sel)])
        return tasks

    def _map(self, fn, args):
        if self.pool is None:
            return [fn(*a) for a in args]
        return self.pool.starmap(fn, args)

    def step(self):
        """One timed step; returns (wall seconds, modelled full-step seconds)."""
        wl = self.wl
        R = wl.B * wl.K
        P = self.P
        cuts = [R * i // P for i in range(P + 1)]
        tasks = self._sample_rows()
        t0 = time.perf_counter()
        self._map(_w_topk, [(cuts[i], cuts[i + 1]) for i in range(P) if cuts[i + 1] > cuts[i]])
        t1 = time.perf_counter()
        self._map(_w_tree, [(b,) for b in range(wl.B)])
        t2 = time.perf_counter()
        attn = self._map(_w_attn, [(rows,) for rows in tasks])
        t3 = time.perf_counter()
        self._map(_w_accept, [(b,) for b in range(wl.B)])
        t4 = time.perf_counter()
        sampled = sum(len(r) for r in tasks)
        attn_full = sum(attn) * self.total_rows / max(1, sampled) / P
        return t4 - t0, (t1 - t0) + (t2 - t1) + (t4 - t3) + attn_full

    def describe(self):
        wl = self.wl
        return (f"per step: oracle stages 1, 2 and 4 on the whole batch ({wl.B * wl.K} drafter rows, {wl.B} trees, "
                f"{int(self.T['n'].sum())} target rows) and attention on {self.ROWS} (node, head) rows from each of "
                f"{min(self.P, len(self.groups))} of the {len(self.groups)} (request, KV head) groups "
                f"({self.total_rows} rows in all); the value is full steps per second under the model: stage 1, 2 "
                f"and 4 wall time plus the sampled attention's CPU time scaled to every row and spread over "
                f"{self.P} cores")


def time_oracle(wl, inp, steps, warmup, seconds=None):
    """The oracle on all host cores (forked pool) plus a one-core figure.
    Must run before this process makes any GPU call.  ``seconds`` (optional)
    bounds the timed loop instead of ``steps``."""
    ob = OracleBench(wl, inp)
    one_wall, one_full = ob.step()           # P = 1, in this process
    P = host_cores()
    ob.start_pool(P)
    try:
        for _ in range(warmup):
            ob.step()
        walls, fulls = [], []
        t_start = time.perf_counter()
        while True:
            w, f = ob.step()
            walls.append(w)
            fulls.append(f)
            if seconds is None and len(walls) >= steps:
                break
            if seconds is not None and time.perf_counter() - t_start >= seconds:
                break
    finally:
        ob.close()
    return {"steps": len(walls), "warmup": warmup, "wall_s": sum(walls), "full_s": sum(fulls),
            "value": len(fulls) / sum(fulls),
            "cores": ob.P, "one_core_value": 1.0 / one_full, "one_core_wall_s": one_wall,
            "sample": ob.describe(), "cpu_model": host_cpu_model()}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    wl = I.WORKLOADS[args.workload]
    inp = I.make_step_inputs(wl, 0)
    r = time_oracle(wl, inp, args.steps, args.warmup)
    value = r["value"]
    cpu = {"value": value, "unit": "steps/s", "cores": r["cores"], "kind": "oracle", "sample": r["sample"],
           "one_core": {"value": r["one_core_value"], "unit": "steps/s", "cores": 1}, "cpu_model": r["cpu_model"]}
    line = {"impl": "reference", "metric": "spec-tree steps/s", "value": value, "unit": "steps/s",
            "n_gpus": world, "steps": r["steps"], "warmup": r["warmup"],
            "ms_per_step": 1000.0 * r["wall_s"] / r["steps"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, "oracle on host cores"), "cpu_baseline": cpu,
            "value_model": "value = timed steps / modelled full-step seconds (stages 1, 2, 4 measured whole, "
                           "attention scaled from a row sample); ms_per_step = measured wall time per timed step",
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu), "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) >= 10:
                        rows.append(p)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        busy = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in busy if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        for r in busy:
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7), ("sw_thermal_slowdown", 8),
                              ("sw_power_cap", 9)):
                if r[col].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "samples_busy": len(busy)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------


def config_of(wl, l2):
    return {"workload": wl.name, "B": wl.B, "K": wl.K, "V": wl.V, "topk": wl.topk, "n_min": wl.n_min,
            "n_max": wl.n_max, "controller": wl.controller, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": wl.d,
            "kv_layout": wl.kv_layout, "ctx": wl.L if wl.L_min == 0 else f"U[{wl.L_min},{wl.L}]",
            "logits": wl.logits, "l2": l2}


def stage_bytes(wl, inp, n):
    """Algorithmic bytes of each stage (every input read once, outputs written once)."""
    es = 2 if wl.dtype == "bf16" else 4
    k1 = wl.B * wl.K * wl.V * es
    kv = 0
    for b in range(wl.B):
        L = int(inp.ctx_len[b])
        nb = int(n[b])
        kv += 2 * wl.Hkv * wl.d * L * es          # context K and V
        kv += 2 * nb * wl.Hkv * wl.d * es         # tree K and V
        kv += 2 * nb * wl.Hq * wl.d * es          # Q in, O out
    k4 = int(sum(int(n[b]) for b in range(wl.B))) * wl.V * es
    return {"topk_softmax": k1, "tree_attn": kv, "accept": k4}


def attn_flops(wl, inp, n, depth):
    """Algorithmic FLOPs of tree attention: for every (node, query head) row,
    Q.K and P.V over the context keys and the node's root-to-node path."""
    f = 0
    for b in range(wl.B):
        L = int(inp.ctx_len[b])
        for i in range(int(n[b])):
            f += wl.Hq * 4 * wl.d * (L + int(depth[b][i]) + 1)
    return f


def step_roofline(sb, flops, hbm_gbs, tensor_tflops, step_us):
    """The step's roofline: the sum of the per-stage minimum times at the peaks
    (each input read once; attention at the larger of its HBM and tensor
    times, HBM alone without a tensor-core count; the tree build, a serial
    chain, has no throughput roofline and counts zero), and that sum over the
    measured step time."""
    t = {"topk_softmax": sb["topk_softmax"] / (hbm_gbs * 1e9), "accept": sb["accept"] / (hbm_gbs * 1e9)}
    t_attn = sb["tree_attn"] / (hbm_gbs * 1e9)
    if flops is not None:
        t_attn = max(t_attn, flops / (tensor_tflops * 1e12))
    t["tree_attn"] = t_attn
    min_us = sum(t.values()) * 1e6
    return {"min_us": min_us, "measured_us": step_us, "frac": min_us / step_us,
            "per_stage_min_us": {k: v * 1e6 for k, v in t.items()}}


def tree_report(step):
    """Per request of the last step run: the chosen tree size n, A_hat(T_n),
    S(n), the accepted length and the tokens the step emits (accepted + bonus)."""
    acc = [int(x) for x in step.acc_len.cpu().numpy()]
    return {"n": [int(x) for x in step.n.cpu().numpy()], "ahat": [float(x) for x in step.ahat.cpu().numpy()],
            "S": [float(x) for x in step.S.cpu().numpy()], "acc_len": acc, "tokens_per_step": [a + 1 for a in acc],
            "mean_tokens_per_step": sum(a + 1 for a in acc) / len(acc)}


def run_ours(args, rank, world, local_rank):
    import torch
    from tree_speculative_decoding_bastion_gb300 import binding as bn
    from tree_speculative_decoding_bastion_gb300 import build

    build.build()
    wl = I.WORKLOADS[args.workload]
    first_set = I.make_step_inputs(wl, replica_seed(rank, 0))
    # ---- CPU baseline: the oracle on the host cores (rank 0, one GPU only),
    # before this process makes any GPU call (its worker pool is forked)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle(wl, first_set, 1, 1, seconds=args.cpu_seconds)
        cpu = {"value": r["value"], "unit": "steps/s", "cores": r["cores"], "kind": "oracle",
               "sample": r["sample"] + f"; {r['steps']} timed steps ({r['wall_s']:.1f} s)",
               "one_core": {"value": r["one_core_value"], "unit": "steps/s", "cores": 1},
               "cpu_model": r["cpu_model"]}
    torch.cuda.set_device(local_rank)
    bn.bastion_init(local_rank)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    hbm, tf_burst, tf_sust, peak_kind = peaks()

    def up(x, bf=False):
        t = torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if bf else x)).cuda()
        return t.view(torch.bfloat16) if bf else t

    bf = wl.dtype == "bf16"

    # ---- input sets, enough to exceed twice the L2
    sets = []
    step = None
    set_bytes = None
    n_sets = args.sets
    r = 0
    while True:
        inp = first_set if r == 0 else I.make_step_inputs(wl, replica_seed(rank, r))
        s = dict(inp=inp, logits=up(inp.logits, bf), root=up(inp.root_tok), ctx=up(inp.ctx_len),
                 C=None if inp.C is None else up(inp.C), q=up(inp.q, bf), kt=up(inp.k_tree, bf),
                 vt=up(inp.v_tree, bf))
        s["kv"] = bn.KV(up(inp.k_ctx, bf), up(inp.v_ctx, bf),
                        None if inp.block_table is None else up(inp.block_table))
        if step is None:
            step = bn.SpecTreeStep(wl.B, wl.K, wl.V, wl.topk, wl.n_min, wl.n_max, wl.Hq, wl.Hkv, wl.d, s["kv"],
                                   act_dtype=dt)
        step.draft(s["logits"], s["root"], s["ctx"], s["C"], inp.L_AR)
        torch.cuda.synchronize()
        depth, n = step.depth.cpu().numpy(), step.n.cpu().numpy()
        s["n"] = n
        s["depth"] = depth
        s["target"] = up(I.make_target_logits(inp, depth, n), bf)
        sets.append(s)
        if set_bytes is None:
            set_bytes = sum(t.numel() * t.element_size() for t in
                            (s["logits"], s["q"], s["kt"], s["vt"], s["kv"].k, s["kv"].v, s["target"]))
            if n_sets <= 0:
                n_sets = max(2, min(16, math.ceil(2 * L2_BYTES / set_bytes)))
        r += 1
        if r >= n_sets:
            break

    def args_of(s):
        return (s["logits"], s["root"], s["ctx"], s["C"], s["inp"].L_AR, s["q"], s["kt"], s["vt"], s["kv"],
                s["inp"].scale, s["target"])

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    # ---- capture one graph per input set
    graphs = []
    with torch.cuda.stream(stream):
        for s in sets:
            step(*args_of(s))
    torch.cuda.synchronize()
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(*args_of(s))
        graphs.append(g)
    # and one graph that runs a step on every input set in turn, so that
    # consecutive steps follow each other inside a graph (programmatic launch
    # between them) instead of paying a graph launch per step
    ring = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ring, stream=stream):
        for s in sets:
            step(*args_of(s))
    torch.cuda.synchronize()
    launches_per_step = 4

    def run_steps(count):
        # exactly `count` steps: whole passes over the sets, then single steps
        for _ in range(count // len(sets)):
            ring.replay()
        for i in range(count % len(sets)):
            graphs[i].replay()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    assert int(step.dev_err.item()) == 0, "device error word set during the benchmark"

    # ---- the same steps launched eagerly: the four calls of every step issued
    # from the host one by one (no graph), the host's launch cost included;
    # each input set's calls are checked and marshalled once (prepare)
    n_eager = min(args.steps, 2000)
    with torch.cuda.stream(stream):
        prepared = [step.prepare(*args_of(s)) for s in sets]
        for i in range(3):
            prepared[i % len(sets)]()
    torch.cuda.synchronize()
    barrier()
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        ev_e[0].record(stream)
        for i in range(n_eager):
            prepared[i % len(sets)]()
        ev_e[1].record(stream)
    torch.cuda.synchronize()
    barrier()
    eager_ms = max_over_ranks(ev_e[0].elapsed_time(ev_e[1]), world)
    assert int(step.dev_err.item()) == 0, "device error word set during the eager steps"
    eager = {"value": job_throughput(world, n_eager, eager_ms), "unit": "steps/s", "steps": n_eager,
             "ms_per_step": eager_ms / n_eager,
             "note": "the same rotating input sets, each step's four library calls launched from the host "
                     "(SpecTreeStep.prepare: arguments checked and marshalled once per input set; programmatic "
                     "launch between the kernels, no CUDA graph); CUDA events on the launching stream"}

    # ---- per-kernel durations: each stage launched back to back over the
    # rotating input sets (2 passes) between two events on the launching
    # stream, the way the stages follow one another inside a step (the
    # programmatic-launch overlap included); mean over 4 repetitions
    names = ("topk_softmax", "tree_build", "tree_attn", "accept")
    s0 = sets[0]

    def launch(kname, s):
        if kname == "topk_softmax":
            bn.bastion_topk_softmax(s["logits"], wl.topk, step.ids, step.lg, step.q, step.lse, dev_err=step.dev_err,
                                    stream=stream)
        elif kname == "tree_build":
            bn.bastion_tree_build(step.ids, step.lg, step.lse, wl.V, s0["root"], s0["ctx"], wl.n_min, wl.n_max,
                                  s0["C"], s0["inp"].L_AR, step.n, step.parent, step.token, step.depth, step.pos,
                                  step.rho, step.mask, step.ahat, step.S, step.S_curve, dev_err=step.dev_err,
                                  stream=stream)
        elif kname == "tree_attn":
            bn.bastion_tree_attn(s["q"], s["kt"], s["vt"], s["kv"], s["ctx"], step.mask, step.n, step.attn_out,
                                 s["inp"].scale, ws=step.attn_ws, dev_err=step.dev_err, stream=stream)
        else:
            bn.bastion_accept(s["target"], step.n, step.parent, step.token, wl.K, step.acc_len, step.acc_nodes,
                              step.acc_tok, step.bonus, step.acc_ws, argmax_out=step.argmax, dev_err=step.dev_err,
                              stream=stream)

    # one step on set 0 so the tree the later stages read belongs to set 0
    with torch.cuda.stream(stream):
        step(*args_of(s0))
    torch.cuda.synchronize()
    per = {k: [] for k in names}
    reps = 2 * len(sets)
    with torch.cuda.stream(stream):
        for kname in names:
            for _ in range(4):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                torch.cuda._sleep(int(10e6))   # keeps the GPU busy while the host queues the launches
                ev[0].record(stream)
                for i in range(reps):
                    launch(kname, sets[(kname == "tree_build") and 0 or (i % len(sets))])
                ev[1].record(stream)
                stream.synchronize()
                per[kname].append(ev[0].elapsed_time(ev[1]) * 1e3 / reps)   # us per launch
    launches_timing = 4 * reps * len(names)
    clk = clocks.stop()
    us = {k: statistics.mean(v) for k, v in per.items()}
    nb = sets[0]["n"]
    sb = stage_bytes(wl, sets[0]["inp"], nb)
    fl = attn_flops(wl, sets[0]["inp"], nb, sets[0]["depth"]) if bf else None

    def roof_of(k):
        t = us[k] * 1e-6
        if k == "tree_attn" and fl is not None and fl / (tf_burst * 1e12) > sb[k] / (hbm * 1e9):
            achieved = fl / t / 1e12
            return {"kernel": k, "bound": "tensor", "achieved": achieved, "peak": tf_burst, "unit": "TFLOP/s",
                    "frac": achieved / tf_burst, "traffic": known_traffic(k, wl.name), "flops_per_launch": fl,
                    "bytes_per_launch": sb[k], "avg_us": us[k], "peak_kind": f"{peak_kind} (burst bf16 GEMM)",
                    "src": kernel_source_hash(k)}
        if k in sb:
            achieved = sb[k] / t / 1e9
            return {"kernel": k, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": known_traffic(k, wl.name), "bytes_per_launch": sb[k],
                    "avg_us": us[k], "peak_kind": f"{peak_kind} (burst copy)", "src": kernel_source_hash(k)}
        return None

    # the dominant kernel among those with a throughput roofline; the serial
    # tree build (one warp per request, a dependent chain of warp reductions)
    # is reported in `stages` with its time and share
    dom = max((k for k in us if k in sb), key=us.get)
    roof = roof_of(dom)
    stages = {}
    for k in names:
        e = {"avg_us": us[k], "share": us[k] / sum(us.values())}
        if k in sb:
            e["GB/s"] = sb[k] / (us[k] * 1e-6) / 1e9
            e["hbm_frac"] = e["GB/s"] / hbm
        if k == "tree_attn" and fl is not None:
            e["TFLOP/s"] = fl / (us[k] * 1e-6) / 1e12
            e["tensor_frac"] = e["TFLOP/s"] / tf_burst
        stages[k] = e

    step_roof = step_roofline(sb, fl, hbm, tf_burst, ms / args.steps * 1e3)
    step_roof["note"] = ("per-stage minimum times at the measured peaks (HBM copy, burst bf16 GEMM) for set 0's "
                         "trees; the tree build counts zero")

    # ---- beyond the step: commit the accepted path of set 0 to a scratch
    # cache laid out like the workload's (contiguous rows with room, or fresh
    # pages for the positions the commit writes), so the workload's own
    # context stays fixed; timed alone, back to back
    commit = None
    if not args.no_commit:
        s = sets[0]
        with torch.cuda.stream(stream):
            step(*args_of(s))
        torch.cuda.synchronize()
        ctx_h = s["ctx"].cpu().numpy()
        acc_h = step.acc_len.cpu().numpy()
        esz = 2 if bf else 4
        if s["inp"].block_table is None:
            shape = (wl.B, wl.Hkv, int(ctx_h.max()) + wl.K + 1, wl.d)
            kv_s = bn.KV(torch.zeros(shape, dtype=dt, device="cuda"), torch.zeros(shape, dtype=dt, device="cuda"))
        else:
            ps = wl.page_size
            cols = (int(ctx_h.max()) + wl.K + ps) // ps
            bt = np.zeros((wl.B, cols), np.int32)
            npg = 0
            for b in range(wl.B):
                for col in range(int(ctx_h[b]) // ps, (int(ctx_h[b]) + wl.K) // ps + 1):
                    bt[b, col] = npg
                    npg += 1
            shape = (npg, wl.Hkv, ps, wl.d)
            kv_s = bn.KV(torch.zeros(shape, dtype=dt, device="cuda"), torch.zeros(shape, dtype=dt, device="cuda"),
                         up(bt))
        ctx_out = torch.empty_like(s["ctx"])

        def commit_once():
            bn.bastion_kv_commit(s["kt"], s["vt"], kv_s, step.acc_len, step.acc_nodes, s["ctx"], ctx_out,
                                 dev_err=step.dev_err, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                commit_once()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda._sleep(int(10e6))
            ev[0].record(stream)
            for _ in range(200):
                commit_once()
            ev[1].record(stream)
        torch.cuda.synchronize()
        assert int(step.dev_err.item()) == 0, "device error word set by the commit"
        assert np.array_equal(ctx_out.cpu().numpy(), ctx_h + acc_h + 1)
        c_us = ev[0].elapsed_time(ev[1]) * 1e3 / 200
        rows = int((acc_h + 1).sum()) * wl.Hkv * 2
        cbytes = rows * wl.d * esz * 2
        commit = {"avg_us": c_us, "rows": rows, "bytes_per_launch": cbytes, "GB/s": cbytes / (c_us * 1e-6) / 1e9,
                  "note": "bastion_kv_commit of set 0's accepted paths (acc_len + 1 rows per request and KV head, "
                          "K and V), bytes read + written; not part of the step"}

    # ---- beyond the step: the drafter's attention over the same context, one
    # block of K mask tokens per request (block-diffusion mask built on the
    # device, then the attention call driven by it); timed alone
    drafter = None
    if not args.no_commit:
        s = sets[0]
        n_blk = torch.full((wl.B,), wl.K, dtype=torch.int32, device="cuda")
        dmask = torch.empty_like(step.mask)
        dout = torch.empty_like(step.attn_out)

        def drafter_once():
            bn.bastion_block_mask(n_blk, wl.K, dmask, dev_err=step.dev_err, stream=stream)
            bn.bastion_tree_attn(s["q"], s["kt"], s["vt"], s["kv"], s["ctx"], dmask, n_blk, dout, s["inp"].scale,
                                 ws=step.attn_ws, dev_err=step.dev_err, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                drafter_once()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda._sleep(int(10e6))
            ev[0].record(stream)
            for _ in range(100):
                drafter_once()
            ev[1].record(stream)
        torch.cuda.synchronize()
        assert int(step.dev_err.item()) == 0, "device error word set by the drafter attention"
        d_us = ev[0].elapsed_time(ev[1]) * 1e3 / 100
        esz = 2 if bf else 4
        ctx_bytes = int(sum(int(x) for x in s["inp"].ctx_len)) * wl.Hkv * wl.d * esz * 2
        drafter = {"avg_us": d_us, "rows": wl.B * wl.K * wl.Hq, "context_bytes": ctx_bytes,
                   "GB/s": ctx_bytes / (d_us * 1e-6) / 1e9,
                   "note": "bastion_block_mask + bastion_tree_attn: B requests x one block of K mask tokens over "
                           "the workload's context (bidirectional inside the block); not part of the step"}

    # ---- beyond the step: stage 2 with the confidence threshold, tau placed
    # at the rho of the middle node of set 0's first tree; timed alone
    pruned = None
    if not args.no_commit:
        s = sets[0]
        with torch.cuda.stream(stream):
            step(*args_of(s))
        torch.cuda.synchronize()
        n0 = int(step.n[0].item())
        tau = float(step.rho[0, max(0, n0 // 2)].item())

        def pruned_once():
            bn.bastion_tree_build(step.ids, step.lg, step.lse, wl.V, s["root"], s["ctx"], 1, wl.n_max, s["C"],
                                  s["inp"].L_AR, step.n, step.parent, step.token, step.depth, step.pos, step.rho,
                                  step.mask, step.ahat, step.S, step.S_curve, dev_err=step.dev_err, stream=stream,
                                  tau=tau)

        with torch.cuda.stream(stream):
            for _ in range(3):
                pruned_once()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda._sleep(int(10e6))
            ev[0].record(stream)
            for _ in range(100):
                pruned_once()
            ev[1].record(stream)
        torch.cuda.synchronize()
        assert int(step.dev_err.item()) == 0, "device error word set by the threshold tree build"
        pruned = {"avg_us": ev[0].elapsed_time(ev[1]) * 1e3 / 100, "tau": tau,
                  "n": [int(x) for x in step.n.cpu().numpy()],
                  "note": "bastion_tree_build_threshold on set 0 with n_min = 1 and tau = rho of the middle node "
                          "of request 0's tree; not part of the step"}
        with torch.cuda.stream(stream):   # the step's own outputs for set 0 again
            step(*args_of(s))
        torch.cuda.synchronize()

    # ---- beyond the step: calibrate the stage-2 cost table on this device
    # (the verification attention timed over N, fitted by the library)
    calib = None
    if not args.no_commit:
        from tree_speculative_decoding_bastion_gb300 import calibrate as cal
        s = sets[0]
        Ns = sorted({1, *[max(1, (wl.n_max * i) // 8) for i in range(1, 9)]})
        t_draft = us["topk_softmax"] + us["tree_build"]
        res = cal.calibrate(s["q"], s["kt"], s["vt"], s["kv"], s["ctx"], s["inp"].scale, Ns, t_draft, reps=20,
                            stream=stream)
        calib = {k: res[k] for k in ("Ns", "t_us", "a", "b", "c", "knee", "rms_us", "t_draft_us", "L_AR")}
        calib["C_n_max"] = float(res["C"][-1].item())
        calib["note"] = ("T_verify(N) = a + b N + c max(0, N - knee) fitted (microseconds) to the tree attention "
                         "timed at each N (bastion_fit_verify_latency); C(n) = t_draft + T_verify(n) with t_draft = "
                         "top-k + tree-build time (bastion_latency_table); not part of the step")

    # ---- end to end through the public API from pinned host buffers: every
    # step copies its whole input block host -> device and its result block
    # back; the runner keeps two slots so one step's copy overlaps the other's
    # compute
    e2e = None
    if not args.no_e2e:
        s = sets[0]
        runner = bn.HostStepRunner(step, s["kv"], s["C"], s["inp"].L_AR, s["inp"].scale, act_dtype=dt, depth=2)
        src = {"logits": s["logits"], "root_tok": s["root"], "ctx_len": s["ctx"], "q": s["q"], "k_tree": s["kt"],
               "v_tree": s["vt"], "target": s["target"]}
        for slot in range(runner.depth):
            for k, v in runner.inputs(slot).items():
                v.copy_(src[k].cpu())
        runner.prepare()
        n_e2e = min(max(args.steps, 20), 4000)
        for _ in range(3):   # warm-up
            runner.submit()
        while runner.in_flight:
            runner.collect()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            runner.submit()
        while runner.in_flight:
            runner.collect()
        t1 = time.perf_counter()
        e2e = {"value": world * n_e2e / (t1 - t0), "unit": "steps/s", "h2d_bytes_per_step": runner.h2d_bytes,
               "d2h_bytes_per_step": runner.d2h_bytes,
               "note": "HostStepRunner, two slots: per step one H2D copy of the step's input block (drafter "
                       "logits, root/ctx ids, tree Q/K/V, target logits) from pinned host memory, the four calls "
                       "(one CUDA graph), one D2H copy of n, accepted length/tokens and bonus; the host waits for "
                       "each result. The context KV cache is resident model state"}

    if rank == 0:
        value = job_throughput(world, args.steps, ms)
        l2 = f"rotating {len(sets)} input sets of {set_bytes / 1e6:.1f} MB (> 2x L2)"
        line = {"metric": "spec-tree steps/s", "value": value, "unit": "steps/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf else "f32",
                "data": "synthetic", "config": config_of(wl, l2), "roofline": roof, "stages": stages,
                "step_roofline": step_roof, "eager": eager,
                "cpu_baseline": cpu, "e2e": e2e, "next_rows": {"kv_commit": commit, "drafter_attention": drafter,
                                                      "tree_build_threshold": pruned,
                                                      "latency_calibration": calib},
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk, "tree": tree_report(step),
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)   # about 2 s timed on long_ctx_b4: the clock sampler sees it
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0 = enough for 2x L2)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-commit", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
