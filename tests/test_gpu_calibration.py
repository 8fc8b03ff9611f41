"""Latency-table calibration on the device: the verification pass timed over
N, the library's fit of those times against the oracle's, and the resulting
table driving the stage-2 controller (bit-exact trees against the oracle with
the same table)."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import calibrate as cal  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402
from .test_gpu_parity import check_tree  # noqa: E402
from .test_gpu_threshold import oracle_tree, run_stage2  # noqa: E402

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


def test_calibrated_table_drives_the_controller():
    wl = W["qwen3_8b_b1"].scaled(name="calib", n_min=1, n_max=256, L=4096)
    inp = I.make_step_inputs(wl, 0)
    kv = C.kv_of(inp)
    Ns = [1, 16, 32, 48, 64, 96, 128, 160, 192, 224, 256]
    res = cal.calibrate(C.dev(inp.q, wl.dtype), C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv,
                        C.dev(inp.ctx_len), inp.scale, Ns, t_draft_us=20.0, reps=10)
    t = np.asarray(res["t_us"])
    assert np.all(np.isfinite(t)) and np.all(t > 0)
    a, b, c, knee, sse = oracle.fit_verify_latency(Ns, t, 1, 256)
    assert res["knee"] == knee
    for g, w in ((res["a"], a), (res["b"], b), (res["c"], c)):
        assert abs(g - w) <= 1e-7 * max(1.0, float(t.max()))
    Cw, L_w = oracle.latency_table(res["a"], res["b"], res["c"], res["knee"], 20.0, 256)
    assert np.array_equal(res["C"].cpu().numpy(), Cw) and res["L_AR"] == L_w
    # the table in the controller: stage 2 on a flat-sweep batch (a smaller
    # vocabulary keeps the oracle quick), against the oracle; the measured
    # table decides how close the S(n+1) vs S(n) comparisons come, so look
    # for a seed without a near tie
    wl2 = W["controller_sweep_flat"].scaled(name="calib_flat", B=2, V=20000)
    for seed in range(40):
        inp2, o2 = C.pick(wl2, seed, with_attention=False)
        inp2 = dataclasses.replace(inp2, C=Cw, L_AR=L_w)
        want = oracle_tree(inp2, o2, 0.0)
        if all(g >= C.GAP for g in want["gaps"]):
            check_tree(run_stage2(inp2, o2, 0.0), want)
            return
    pytest.skip("no seed without a near tie under the calibrated table")
