"""Calibration of the stage-2 cost table C(N) on the current device.

BASTION page ("Bastion: Budget-Aware Speculative Decoding with
Tree-structured Block Diffusion Drafting"), Methodik §3: the online controller
needs C(N), the cost of a step that verifies N tree tokens, and L_AR; the
pages model the verification latency from memory bandwidth and compute,
calibrated on the device's observed runtimes.

Here the verification pass is this library's tree attention: it is timed with
CUDA events at several tree sizes N (every request's tree of size N, its mask
built on the device by bastion_block_mask -- the kernel's cost does not depend
on which mask bits are set), the times are fitted with the library's
bastion_fit_verify_latency, and bastion_latency_table turns the fit plus the
caller's drafting time into the table bastion_tree_build takes.  Timing and
marshalling only: the attention, the mask and the fit run in the library.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import binding as bn


def measure_verify_us(q, k_tree, v_tree, kv: bn.KV, ctx_len, scale: float, Ns: Sequence[int], reps: int = 20,
                      stream: Optional[torch.cuda.Stream] = None) -> np.ndarray:
    """Mean microseconds of one bastion_tree_attn call with n[b] = N for every
    request, for each N in Ns (N <= q.shape[1]); `reps` back-to-back launches
    per N after three warm-up calls, timed with CUDA events on `stream`."""
    B, n_max, Hq, d = q.shape
    Hkv = k_tree.shape[2]
    if max(Ns) > n_max or min(Ns) < 1:
        raise bn.BastionError(f"every N must lie in [1, {n_max}]")
    st = torch.cuda.current_stream() if stream is None else stream
    out = torch.empty_like(q)
    mask = torch.empty(B, n_max, (n_max + 63) // 64, dtype=torch.int64, device=q.device)
    ws = torch.zeros(max(1, bn.bastion_tree_attn_workspace_size(B, n_max, Hq, Hkv, d, kv)), dtype=torch.uint8,
                     device=q.device)
    err = torch.zeros(1, dtype=torch.int32, device=q.device)
    times = []
    with torch.cuda.stream(st):
        for N in Ns:
            n = torch.full((B,), int(N), dtype=torch.int32, device=q.device)
            bn.bastion_block_mask(n, int(N), mask, dev_err=err, stream=st)
            for _ in range(3):
                bn.bastion_tree_attn(q, k_tree, v_tree, kv, ctx_len, mask, n, out, scale, ws=ws, dev_err=err,
                                     stream=st)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(reps):
                bn.bastion_tree_attn(q, k_tree, v_tree, kv, ctx_len, mask, n, out, scale, ws=ws, dev_err=err,
                                     stream=st)
            e1.record(st)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / reps)
    if int(err.item()) != 0:
        raise bn.BastionError(f"device error word {int(err.item()):#x} while timing the verification pass")
    return np.asarray(times, dtype=np.float64)


def calibrate(q, k_tree, v_tree, kv: bn.KV, ctx_len, scale: float, Ns: Sequence[int], t_draft_us: float,
              knee_lo: int = 1, knee_hi: Optional[int] = None, reps: int = 20,
              stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Time the verification pass at each N, fit T_verify(N), and build the
    stage-2 table for n_max = q.shape[1].  Returns a dict with the measured
    points (Ns, t_us), the fit (a, b, c, knee, sse, rms_us), L_AR and C (a
    float32 CUDA tensor of n_max + 1 entries, microseconds)."""
    n_max = q.shape[1]
    t = measure_verify_us(q, k_tree, v_tree, kv, ctx_len, scale, Ns, reps=reps, stream=stream)
    hi = n_max if knee_hi is None else knee_hi
    a, b, c, knee, sse = bn.bastion_fit_verify_latency(np.asarray(Ns), t, knee_lo, hi)
    C, L_AR = bn.bastion_latency_table(a, b, c, knee, t_draft_us, n_max)
    return {"Ns": [int(x) for x in Ns], "t_us": [float(x) for x in t], "a": a, "b": b, "c": c, "knee": knee,
            "sse": sse, "rms_us": float(np.sqrt(sse / len(Ns))), "t_draft_us": float(t_draft_us), "L_AR": L_AR,
            "C": torch.from_numpy(C).to(q.device)}
