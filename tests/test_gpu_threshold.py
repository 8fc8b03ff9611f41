"""Stage 2 with the confidence threshold (bastion_tree_build_threshold) against
the oracle: bit-exact trees, with a fixed budget and with the S(N)
controller.  tau is placed between two consecutive nodes' rho of the first
request, and only where no request has a node within the near-tie gap of it."""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402
from .test_gpu_parity import SMALL, check_tree  # noqa: E402

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


CASES = {
    "qwen3_fixed_nmin8": W["qwen3_8b_b1"].scaled(name="qwen3_tau", n_min=8),
    "flat_controller": W["controller_sweep_flat"],
    "peaked_controller": W["controller_sweep_peaked"],
    "ragged_fixed": SMALL["qwen3_ragged"].scaled(name="ragged_tau", n_min=20),
    "tiny_f32": W["tiny_v1024_f32"].scaled(name="tiny_tau", n_min=4),
}


def oracle_tree(inp, o, tau):
    wl = inp.wl
    B, K = wl.B, wl.K
    trees = oracle.tree_build(o["ids"].reshape(B, K, -1), o["lg"].reshape(B, K, -1), o["lse"].reshape(B, K),
                              inp.root_tok, inp.ctx_len, wl.n_min, wl.n_max, inp.C, inp.L_AR, tau)
    return oracle.stack_trees(trees)


def pick_tau(inp, o):
    """A tau strictly between two consecutive nodes of request 0 (past n_min),
    with every request's decisions clear of the near-tie gap."""
    wl = inp.wl
    rho = o["tree"]["rho"][0][: int(o["tree"]["n"][0])]
    for m in list(range(max(wl.n_min + 1, len(rho) // 2), len(rho))) + list(range(wl.n_min + 1, len(rho) // 2)):
        if not rho[m - 1] > rho[m] * 1.01:
            continue
        tau = math.sqrt(rho[m - 1] * rho[m])
        t = oracle_tree(inp, o, tau)
        if all(g >= C.GAP for g in t["gaps"]):
            return tau, t
    pytest.skip("no threshold clear of every near tie")


def run_stage2(inp, o, tau):
    wl = inp.wl
    B, K, k, N = wl.B, wl.K, wl.topk, wl.n_max
    ids = C.dev(o["ids"].reshape(B, K, k).astype(np.int32))
    lg = C.dev(o["lg"].reshape(B, K, k).astype(np.float32))
    lse = C.dev(o["lse"].reshape(B, K).astype(np.float64))
    t = dict(n=torch.empty(B, dtype=torch.int32, device="cuda"))
    for name in ("parent", "token", "depth", "pos"):
        t[name] = torch.empty(B, N, dtype=torch.int32, device="cuda")
    t["rho"] = torch.empty(B, N, dtype=torch.float32, device="cuda")
    t["mask"] = torch.empty(B, N, (N + 63) // 64, dtype=torch.int64, device="cuda")
    t["ahat"] = torch.empty(B, dtype=torch.float32, device="cuda")
    t["S"] = torch.empty(B, dtype=torch.float32, device="cuda")
    t["S_curve"] = torch.empty(B, N, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ct = None if inp.C is None else C.dev(inp.C)
    bn.bastion_tree_build(ids, lg, lse, wl.V, C.dev(inp.root_tok), C.dev(inp.ctx_len), wl.n_min, N, Ct, inp.L_AR,
                          t["n"], t["parent"], t["token"], t["depth"], t["pos"], t["rho"], t["mask"], t["ahat"],
                          t["S"], t["S_curve"], dev_err=err, tau=tau)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {k_: v.cpu().numpy() for k_, v in t.items()}


@pytest.mark.parametrize("name", list(CASES))
def test_threshold_tree_matches_oracle(name):
    wl = CASES[name]
    inp, o = C.pick(wl, 0, with_attention=False)
    tau, want = pick_tau(inp, o)
    assert want["n"][0] < o["tree"]["n"][0] or wl.n_min == o["tree"]["n"][0]   # the threshold cut request 0
    got = run_stage2(inp, o, tau)
    check_tree(got, want)
    # a threshold above every node: each request keeps n_min nodes (or fewer if its tree is smaller)
    got = run_stage2(inp, o, 1.0)
    assert np.array_equal(got["n"], np.minimum(wl.n_min, o["tree"]["n"]))
