"""Seeded synthetic workloads for the spec-tree step.

This module only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no softmax over drafter rows, no tree search, no attention,
no argmax), so both the CUDA path and the CPU oracle can consume what it makes.

Every array is numpy.  bf16 tensors are carried as ``uint16`` bit patterns,
rounded to nearest-even from float32, so the CUDA side and the oracle read
exactly the same values.

Workload shapes follow the BASTION explainer pages (gist.science 2605.29727,
"Technische Zusammenfassung" / "Experimentelle Ergebnisse"): a Qwen3-8B-shaped
target (V=151936, 32 query / 8 KV heads, head_dim 128) and a Llama-3.1-8B-shaped
one (V=128256), greedy decoding, block-diffusion drafter with K positions.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# --------------------------------------------------------------------------
# bf16 bit helpers (a dtype cast, not method arithmetic)
# --------------------------------------------------------------------------


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored tensor (float32 or bf16 bits) -> float32 values."""
    return bf16_bits_to_f32(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> the stored form for ``dtype``."""
    return to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # requests
    K: int                 # drafter block positions (max tree depth)
    V: int                 # vocabulary
    topk: int              # candidates per position
    n_min: int             # controller lower bound on tree size (root included)
    n_max: int             # tree budget cap N_max (root included)
    controller: bool       # False: fixed budget, no latency table
    dtype: str             # "f32" or "bf16" for logits / Q / K / V
    Hq: int
    Hkv: int
    d: int
    kv_layout: str         # "contiguous" or "paged"
    L: int                 # fixed context length (contiguous), or max of the range
    L_min: int = 0         # >0: per-request context drawn uniformly in [L_min, L]
    page_size: int = 16
    logits: str = "planted"   # "planted" | "normal_planted_range" | "peaked" | "flat"
    logit_sigma: float = 1.0
    plant: float = 4.0        # planted offset (fixed) for "planted"
    plant_lo: float = 3.0     # planted offset range for "normal_planted_range"
    plant_hi: float = 8.0
    target_sigma: float = 0.5

    @property
    def rows(self) -> int:
        return self.B * self.K

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (reduced sizes for quick oracle runs)."""
        return dataclasses.replace(self, **kw)


# The five workloads of the spec-tree step.  Names say what they are.
WORKLOADS = {
    # tiny correctness case: fp32, one head, fixed budget 16
    "tiny_v1024_f32": Workload(
        name="tiny_v1024_f32", B=1, K=4, V=1024, topk=4, n_min=16, n_max=16,
        controller=False, dtype="f32", Hq=1, Hkv=1, d=64, kv_layout="contiguous",
        L=128, logits="planted", logit_sigma=1.0, plant=4.0, target_sigma=0.5),
    # Qwen3-8B-shaped single request, fixed budget 64
    "qwen3_8b_b1": Workload(
        name="qwen3_8b_b1", B=1, K=16, V=151936, topk=8, n_min=64, n_max=64,
        controller=False, dtype="bf16", Hq=32, Hkv=8, d=128, kv_layout="contiguous",
        L=4096, logits="normal_planted_range", logit_sigma=2.0, plant_lo=3.0, plant_hi=8.0,
        target_sigma=1.0),
    # Llama-3.1-8B-shaped batch of 16, paged KV, S(N) controller in [8, 64]
    "llama31_8b_b16_paged": Workload(
        name="llama31_8b_b16_paged", B=16, K=16, V=128256, topk=8, n_min=8, n_max=64,
        controller=True, dtype="bf16", Hq=32, Hkv=8, d=128, kv_layout="paged",
        L=8192, L_min=512, page_size=16, logits="planted", logit_sigma=1.0, plant=4.0,
        target_sigma=0.5),
    # long context, 4 requests x 32768 tokens, fixed budget 128
    "long_ctx_b4": Workload(
        name="long_ctx_b4", B=4, K=16, V=151936, topk=8, n_min=128, n_max=128,
        controller=False, dtype="bf16", Hq=32, Hkv=8, d=128, kv_layout="contiguous",
        L=32768, logits="planted", logit_sigma=1.0, plant=4.0, target_sigma=0.5),
    # controller sweep, peaked drafter (top-1 probability about 0.9)
    "controller_sweep_peaked": Workload(
        name="controller_sweep_peaked", B=8, K=16, V=151936, topk=16, n_min=1, n_max=256,
        controller=True, dtype="bf16", Hq=32, Hkv=8, d=128, kv_layout="contiguous",
        L=2048, logits="peaked", target_sigma=1.0),
    # controller sweep, flat drafter (top-1 probability about 0.3)
    "controller_sweep_flat": Workload(
        name="controller_sweep_flat", B=8, K=16, V=151936, topk=16, n_min=1, n_max=256,
        controller=True, dtype="bf16", Hq=32, Hkv=8, d=128, kv_layout="contiguous",
        L=2048, logits="flat", target_sigma=1.0),
}


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), *[int(s) for s in stream]]))


def _drafter_row(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    """One drafter position's logits over the vocabulary (float32)."""
    V = wl.V
    z = rng.standard_normal(V, dtype=np.float32)
    if wl.logits == "planted":
        x = z * np.float32(wl.logit_sigma)
        t = int(rng.integers(V))
        x[t] += np.float32(wl.plant)
        return x
    if wl.logits == "normal_planted_range":
        x = z * np.float32(wl.logit_sigma)
        t = int(rng.integers(V))
        x[t] += np.float32(rng.uniform(wl.plant_lo, wl.plant_hi))
        return x
    if wl.logits == "peaked":
        # Plant one token so that its probability is about 0.9.  For N(0,1)
        # noise the bulk mass sum_u e^{z_u} concentrates at V*e^{1/2}; an offset
        # of ln 9 + ln V + 1/2 puts the planted token at odds 9:1 against the bulk.
        t = int(rng.integers(V))
        x = z.copy()
        x[t] += np.float32(np.log(9.0) + np.log(V) + 0.5)
        return x
    if wl.logits == "flat":
        return z   # scaled by a per-row temperature in flat_rows()
    raise ValueError(f"unknown logit regime {wl.logits!r}")


def flat_rows(z: np.ndarray) -> np.ndarray:
    """Per-row temperature T (bisection on log T, all rows at once) so that the
    largest share e^{z_max/T} / sum_u e^{z_u/T} is 0.30; returns z / T.  This
    calibrates the input only."""
    z = np.asarray(z, dtype=np.float32)
    d = z - z.max(axis=1, keepdims=True)
    lo = np.full((z.shape[0], 1), np.log(1e-3), dtype=np.float32)
    hi = np.full((z.shape[0], 1), np.log(10.0), dtype=np.float32)
    for _ in range(26):
        mid = 0.5 * (lo + hi)
        share = 1.0 / np.exp(d / np.exp(mid)).sum(axis=1, keepdims=True)
        too_peaked = share > 0.30
        lo = np.where(too_peaked, mid, lo)
        hi = np.where(too_peaked, hi, mid)
    return (z / np.exp(0.5 * (lo + hi))).astype(np.float32)


@dataclass
class StepInputs:
    """Everything one spec-tree step reads (numpy, host)."""
    wl: Workload
    seed: int
    logits: np.ndarray            # [B, K, V] float32 or bf16 bits
    root_tok: np.ndarray          # [B] int32
    ctx_len: np.ndarray           # [B] int32
    C: Optional[np.ndarray]       # [n_max + 1] float32, C[n] for n = 1..n_max; None = fixed budget
    L_AR: float
    q: np.ndarray                 # [B, n_max, Hq, d]
    k_tree: np.ndarray            # [B, n_max, Hkv, d]
    v_tree: np.ndarray            # [B, n_max, Hkv, d]
    k_ctx: np.ndarray             # contiguous [B, Hkv, L, d] | paged [P, Hkv, page, d]
    v_ctx: np.ndarray
    block_table: Optional[np.ndarray] = None   # paged: [B, max_pages] int32
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.wl.d))


def latency_table(wl: Workload, seed: int):
    """Per-N cost table C(N) = T_draft + T_verify(N), T_verify(N) = a + bN + c max(0, N-64).

    The constants are seeded draws (arbitrary time units); L_AR = T_verify(1).
    Returns (C[n_max+1] float32 with C[0] = C[1], L_AR) or (None, 1.0) for a fixed budget.
    """
    if not wl.controller:
        return None, 1.0
    r = _rng(seed, 7)
    a = r.uniform(4.0, 8.0)
    b = r.uniform(0.01, 0.05)
    c = r.uniform(0.05, 0.2)
    t_draft = r.uniform(0.5, 1.5)
    N = np.arange(wl.n_max + 1, dtype=np.float64)
    t_verify = a + b * N + c * np.maximum(0.0, N - 64.0)
    C = (t_draft + t_verify).astype(np.float32)
    C[0] = C[1]
    L_AR = float(np.float32(a + b * 1.0))
    return C, L_AR


def make_step_inputs(wl: Workload, seed: int, *, with_attention: bool = True,
                     req_seeds: Optional[tuple] = None) -> StepInputs:
    """Draw every input of one step for workload ``wl`` from ``seed``.

    ``req_seeds[b]`` (optional) replaces ``seed`` for request b's drafter
    logits only, so one request can be redrawn without touching the others.
    """
    B, K, V = wl.B, wl.K, wl.V
    logits32 = np.empty((B, K, V), dtype=np.float32)
    for b in range(B):
        sb = seed if req_seeds is None else int(req_seeds[b])
        for k in range(K):
            logits32[b, k] = _drafter_row(wl, _rng(sb, 1, b, k))
    if wl.logits == "flat":
        logits32 = flat_rows(logits32.reshape(B * K, V)).reshape(B, K, V)
    r = _rng(seed, 2)
    root_tok = r.integers(0, V, size=B).astype(np.int32)
    if wl.L_min > 0:
        ctx_len = r.integers(wl.L_min, wl.L + 1, size=B).astype(np.int32)
    else:
        ctx_len = np.full(B, wl.L, dtype=np.int32)
    C, L_AR = latency_table(wl, seed)

    N, Hq, Hkv, d = wl.n_max, wl.Hq, wl.Hkv, wl.d
    block_table = None
    if with_attention:
        ra = _rng(seed, 3)
        q = ra.standard_normal((B, N, Hq, d), dtype=np.float32)
        k_tree = ra.standard_normal((B, N, Hkv, d), dtype=np.float32)
        v_tree = ra.standard_normal((B, N, Hkv, d), dtype=np.float32)
        rk = _rng(seed, 4)
        if wl.kv_layout == "contiguous":
            Lmax = int(ctx_len.max())
            k_ctx = rk.standard_normal((B, Hkv, Lmax, d), dtype=np.float32)
            v_ctx = rk.standard_normal((B, Hkv, Lmax, d), dtype=np.float32)
        else:
            ps = wl.page_size
            npages = [(int(L) + ps - 1) // ps for L in ctx_len]
            P = int(sum(npages))
            max_pages = (wl.L + ps - 1) // ps
            perm = rk.permutation(P).astype(np.int32)
            block_table = np.full((B, max_pages), -1, dtype=np.int32)
            o = 0
            for b in range(B):
                block_table[b, : npages[b]] = perm[o : o + npages[b]]
                o += npages[b]
            k_ctx = rk.standard_normal((P, Hkv, ps, d), dtype=np.float32)
            v_ctx = rk.standard_normal((P, Hkv, ps, d), dtype=np.float32)
        q, k_tree, v_tree = (store(x, wl.dtype) for x in (q, k_tree, v_tree))
        k_ctx, v_ctx = store(k_ctx, wl.dtype), store(v_ctx, wl.dtype)
    else:
        empty = np.zeros((0,), dtype=np.float32)
        q = k_tree = v_tree = k_ctx = v_ctx = empty
    return StepInputs(wl=wl, seed=seed, logits=store(logits32, wl.dtype), root_tok=root_tok,
                      ctx_len=ctx_len, C=C, L_AR=L_AR, q=q, k_tree=k_tree, v_tree=v_tree,
                      k_ctx=k_ctx, v_ctx=v_ctx, block_table=block_table,
                      extra={"req_seeds": None if req_seeds is None else tuple(int(x) for x in req_seeds)})


def make_target_logits(inp: StepInputs, depth: np.ndarray, n: np.ndarray) -> np.ndarray:
    """Target logits standing in for the target model's LM head.

    Row (b, i) for a tree node at depth d is the drafter's logits at position
    min(d+1, K) (1-based) plus N(0, sigma) noise drawn from its own stream, so
    the target's greedy token usually agrees with the drafter's top-1.  Rows
    i >= n[b] are zero.  ``depth`` is [B, n_max] int; only rows < n[b] are used.
    """
    wl = inp.wl
    B, V, N = wl.B, wl.V, wl.n_max
    drafter = as_f32(inp.logits, wl.dtype)
    out = np.zeros((B, N, V), dtype=np.float32)
    for b in range(B):
        for i in range(int(n[b])):
            pos = min(int(depth[b, i]) + 1, wl.K) - 1
            noise = _rng(inp.seed, 5, b, i).standard_normal(V, dtype=np.float32)
            out[b, i] = drafter[b, pos] + np.float32(wl.target_sigma) * noise
    return store(out, wl.dtype)
