"""The algorithmic bytes and FLOPs behind bench.py's roofline line, checked
against the counts written out by hand for the Qwen3-8B-shaped B=1 workload
(every input read once, outputs written once)."""
import importlib.util
import os

import numpy as np

from tree_speculative_decoding_bastion_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


class _Inp:
    def __init__(self, ctx):
        self.ctx_len = np.asarray(ctx, np.int32)


def test_stage_bytes_by_hand():
    wl = I.WORKLOADS["qwen3_8b_b1"]
    sb = bench().stage_bytes(wl, _Inp([4096]), np.array([64]))
    assert sb["topk_softmax"] == 1 * 16 * 151936 * 2                 # drafter logits, bf16
    ctx = 2 * 8 * 128 * 4096 * 2                                      # context K and V
    tree = 2 * 64 * 8 * 128 * 2                                       # tree K and V
    qo = 2 * 64 * 32 * 128 * 2                                        # Q in, O out
    assert sb["tree_attn"] == ctx + tree + qo == 18087936
    assert sb["accept"] == 64 * 151936 * 2                            # target rows of the 64 nodes


def test_attention_flops_by_hand():
    wl = I.WORKLOADS["qwen3_8b_b1"].scaled(B=2)
    n = np.array([3, 2])
    depth = [np.array([0, 1, 2, -1]), np.array([0, 1, -1, -1])]
    f = bench().attn_flops(wl, _Inp([10, 7]), n, depth)
    # per (node, query head): 2 d flops for Q.K and 2 d for P.V per visible key
    per_key = 32 * 4 * 128
    keys = (10 + 1) + (10 + 2) + (10 + 3) + (7 + 1) + (7 + 2)
    assert f == per_key * keys


def test_step_roofline_sums_the_stage_minima():
    # 1 GB/s and 1 TFLOP/s peaks make every minimum time readable by eye
    sb = {"topk_softmax": 2000, "tree_attn": 3000, "accept": 5000}
    b = bench()
    r = b.step_roofline(sb, None, 1.0, 1.0, 20.0)             # no tensor count: attention at HBM
    assert r["per_stage_min_us"] == {"topk_softmax": 2.0, "accept": 5.0, "tree_attn": 3.0}
    assert r["min_us"] == 10.0 and r["frac"] == 0.5
    r = b.step_roofline(sb, 7e6, 1.0, 1.0, 20.0)              # 7 us of tensor work binds attention
    assert r["per_stage_min_us"]["tree_attn"] == 7.0 and r["min_us"] == 14.0
    r = b.step_roofline(sb, 1e6, 1.0, 1.0, 20.0)              # 1 us of tensor work: HBM still binds
    assert r["per_stage_min_us"]["tree_attn"] == 3.0
