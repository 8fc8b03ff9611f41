"""Parity of the CUDA path with the CPU oracle, stage by stage and end to end.

Bars (from the workload's definition): tree structure, tokens, masks,
argmax and accepted paths bit-exact; probabilities (q, rho, A_hat, S) within
1e-5 relative; attention within 2e-2 absolute + 1e-2 relative for bf16 and
1e-4 for the fp32 path.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402

RTOL_P = 1e-5

W = I.WORKLOADS
# small variants that still span several tiles and ragged tails
SMALL = {
    "qwen3_ragged": W["qwen3_8b_b1"].scaled(name="qwen3_ragged", B=2, V=20000, L=1000, n_min=200, n_max=200,
                                             Hq=16, Hkv=4),
    "paged_ragged": W["llama31_8b_b16_paged"].scaled(name="paged_ragged", B=3, V=9000, L=700, L_min=130,
                                                     n_min=8, n_max=64),
    "unaligned_vocab": W["tiny_v1024_f32"].scaled(name="unaligned_vocab", B=2, V=1001, K=5, topk=7, n_min=40,
                                                  n_max=40, L=77),
    "unaligned_bf16": W["qwen3_8b_b1"].scaled(name="unaligned_bf16", B=1, V=5003, K=8, n_min=48, n_max=48, L=200),
    "mha_d64": W["qwen3_8b_b1"].scaled(name="mha_d64", B=2, V=4096, K=6, topk=4, n_min=30, n_max=30, Hq=2, Hkv=2,
                                       d=64, L=300),
    # CTA pairs over paged caches: 64-key halves made of 8-, 32- or 64-token
    # pages; 128-token pages take the single-CTA form; three M-tiles (the
    # second pair half empty)
    "paged_p8": W["llama31_8b_b16_paged"].scaled(name="paged_p8", B=2, V=4096, L=500, L_min=100, page_size=8,
                                                 n_min=40, n_max=40),
    "paged_p32": W["llama31_8b_b16_paged"].scaled(name="paged_p32", B=2, V=4096, L=700, L_min=90, page_size=32,
                                                  n_min=80, n_max=96),
    "paged_p64": W["llama31_8b_b16_paged"].scaled(name="paged_p64", B=2, V=4096, L=900, L_min=300, page_size=64,
                                                  n_min=60, n_max=64),
    "paged_p128": W["llama31_8b_b16_paged"].scaled(name="paged_p128", B=2, V=4096, L=800, L_min=129, page_size=128,
                                                   n_min=50, n_max=64),
    "three_mtiles": W["qwen3_8b_b1"].scaled(name="three_mtiles", B=2, V=4096, K=8, L=333, n_min=96, n_max=96),
}
FULL = ["tiny_v1024_f32", "qwen3_8b_b1", "llama31_8b_b16_paged", "long_ctx_b4", "controller_sweep_peaked",
        "controller_sweep_flat"]
ALL = {**{k: W[k] for k in FULL}, **SMALL}


@pytest.fixture(scope="session", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


def relclose(a, b, rtol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b) / np.maximum(np.abs(b), 1e-30)
    assert np.all(err <= rtol), f"{what}: max rel err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}"


def run_draft(inp):
    wl = inp.wl
    B, K, k, N = wl.B, wl.K, wl.topk, wl.n_max
    logits = C.dev(inp.logits, wl.dtype)
    out = dict(ids=torch.empty(B, K, k, dtype=torch.int32, device="cuda"),
               lg=torch.empty(B, K, k, dtype=torch.float32, device="cuda"),
               q=torch.empty(B, K, k, dtype=torch.float32, device="cuda"),
               lse=torch.empty(B, K, dtype=torch.float64, device="cuda"))
    bn.bastion_topk_softmax(logits, k, out["ids"], out["lg"], out["q"], out["lse"])
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
    bn.bastion_tree_build(out["ids"], out["lg"], out["lse"], wl.V, C.dev(inp.root_tok), C.dev(inp.ctx_len), wl.n_min,
                          N, Ct, inp.L_AR, t["n"], t["parent"], t["token"], t["depth"], t["pos"], t["rho"], t["mask"],
                          t["ahat"], t["S"], t["S_curve"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {k_: v.cpu().numpy() for k_, v in out.items()}, {k_: v.cpu().numpy() for k_, v in t.items()}


def check_stage1(wl, got, want):
    R = wl.B * wl.K
    assert np.array_equal(got["ids"].reshape(R, -1), want["ids"])
    assert np.array_equal(got["lg"].reshape(R, -1).astype(np.float64), want["lg"])
    relclose(got["q"].reshape(R, -1), want["q"], RTOL_P, "q")
    assert np.all(np.abs(got["lse"].reshape(R) - want["lse"]) <= 1e-5), "lse"


def check_tree(got, want):
    for k_ in ("n", "parent", "token", "depth", "pos"):
        assert np.array_equal(got[k_], want[k_]), k_
    assert np.array_equal(got["mask"].view(np.uint64), want["mask"]), "mask"
    relclose(got["rho"], want["rho"], RTOL_P, "rho")
    relclose(got["ahat"], want["ahat"], RTOL_P, "ahat")
    relclose(got["S"], want["S"], RTOL_P, "S")
    relclose(got["S_curve"], want["S_curve"], RTOL_P, "S_curve")


@pytest.mark.parametrize("name", list(ALL))
def test_draft_stages_match_oracle(name):
    wl = ALL[name]
    inp, o = C.pick(wl, 0, with_attention=False)
    s1, tree = run_draft(inp)
    check_stage1(wl, s1, o)
    check_tree(tree, o["tree"])


@pytest.mark.parametrize("name", ["tiny_v1024_f32", "qwen3_8b_b1", "controller_sweep_flat", "paged_ragged"])
def test_tree_build_from_oracle_stage1(name):
    """Stage 2 alone, fed the oracle's stage-1 table."""
    wl = ALL[name]
    inp, o = C.pick(wl, 0, with_attention=False)
    B, K, k, N = wl.B, wl.K, wl.topk, wl.n_max
    ids = torch.from_numpy(o["ids"].reshape(B, K, k)).cuda()
    lg = torch.from_numpy(o["lg"].reshape(B, K, k).astype(np.float32)).cuda()
    lse = torch.from_numpy(o["lse"].reshape(B, K)).cuda()
    t = {n_: torch.empty(B, N, dtype=torch.int32, device="cuda") for n_ in ("parent", "token", "depth", "pos")}
    t["n"] = torch.empty(B, dtype=torch.int32, device="cuda")
    t["rho"] = torch.empty(B, N, dtype=torch.float32, device="cuda")
    t["mask"] = torch.empty(B, N, (N + 63) // 64, dtype=torch.int64, device="cuda")
    t["ahat"] = torch.empty(B, dtype=torch.float32, device="cuda")
    t["S"] = torch.empty(B, dtype=torch.float32, device="cuda")
    t["S_curve"] = torch.empty(B, N, dtype=torch.float32, device="cuda")
    Ct = None if inp.C is None else C.dev(inp.C)
    bn.bastion_tree_build(ids, lg, lse, wl.V, C.dev(inp.root_tok), C.dev(inp.ctx_len), wl.n_min, N, Ct, inp.L_AR,
                          t["n"], t["parent"], t["token"], t["depth"], t["pos"], t["rho"], t["mask"], t["ahat"],
                          t["S"], t["S_curve"])
    check_tree({k_: v.cpu().numpy() for k_, v in t.items()}, o["tree"])


def attn_tol(wl):
    return (2e-2, 1e-2) if wl.dtype == "bf16" else (1e-4, 1e-4)


def _attention_parity(inp, tree, max_rows, kv=None, rows=None):
    wl = inp.wl
    kv = C.kv_of(inp) if kv is None else kv
    out = torch.full((wl.B, wl.n_max, wl.Hq, wl.d), float("nan"), device="cuda",
                     dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32)
    ws = torch.zeros(max(1, bn.bastion_tree_attn_workspace_size(wl.B, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv)),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_tree_attn(C.dev(inp.q, wl.dtype), C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv,
                         C.dev(inp.ctx_len), C.dev(tree["mask"].view(np.int64)), C.dev(tree["n"]), out, inp.scale,
                         ws=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.float().cpu().numpy()
    total = int(tree["n"].sum()) * wl.Hq
    if rows is None and total > max_rows:
        rows = C.attention_rows(inp, tree, max_rows)
    want = C.oracle_attention(inp, tree, rows=rows)
    if rows is None:
        rows = [(b, i, h) for b in range(wl.B) for i in range(int(tree["n"][b])) for h in range(wl.Hq)]
    atol, rtol = attn_tol(wl)
    g = np.stack([got[r] for r in rows])
    w = np.stack([want[r] for r in rows])
    bad = np.abs(g - w) > atol + rtol * np.abs(w)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; max err {np.abs(g - w).max():.3g}"
    # rows past n[b] are left untouched
    for b in range(wl.B):
        assert np.isnan(got[b, int(tree["n"][b]):]).all()


@pytest.mark.parametrize("name", list(SMALL))
def test_tree_attention_matches_oracle(name):
    """Stage 3 alone on the oracle's tree, every (node, head) row compared."""
    wl = ALL[name]
    inp, o = C.pick(wl, 0)
    _attention_parity(inp, o["tree"], max_rows=1 << 30)


@pytest.mark.parametrize("name", list(ALL))
def test_accept_matches_oracle(name):
    wl = ALL[name]
    inp, o = C.pick(wl, 0, with_attention=False)
    tree = o["tree"]
    target = C.target_for(inp, tree)
    want = C.oracle_accept(inp, tree, target)
    B, N, K = wl.B, wl.n_max, wl.K
    res = {k_: torch.empty(*s, dtype=torch.int32, device="cuda")
           for k_, s in (("acc_len", (B,)), ("acc_nodes", (B, K + 1)), ("acc_tok", (B, K + 1)), ("bonus", (B,)),
                         ("argmax", (B, N)))}
    ws = torch.zeros(bn.bastion_accept_workspace_size(B, N), dtype=torch.uint8, device="cuda")
    tgt = C.dev(target, wl.dtype)
    for rep in range(2):   # the workspace's ticket words return to zero
        bn.bastion_accept(tgt, C.dev(tree["n"]), C.dev(tree["parent"]), C.dev(tree["token"]), K, res["acc_len"],
                          res["acc_nodes"], res["acc_tok"], res["bonus"], ws, argmax_out=res["argmax"])
        torch.cuda.synchronize()
        got = {k_: v.cpu().numpy() for k_, v in res.items()}
        for k_, wv in zip(("acc_len", "acc_nodes", "acc_tok", "bonus", "argmax"), want):
            assert np.array_equal(got[k_], wv), (k_, rep)
    assert (ws == 0).all()   # tickets and row slots are zero again


@pytest.mark.parametrize("name", FULL)
def test_attention_and_whole_step_match_oracle(name):
    """At the workload's full size: stage 3 alone on the oracle's tree (sampled
    rows), then the four calls on device buffers, one stream, no host sync
    between, twice in a row on the same workspaces."""
    wl = W[name]
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    kv = C.kv_of(inp)
    _attention_parity(inp, tree, max_rows=96, kv=kv)
    target = C.target_for(inp, tree)
    step = bn.SpecTreeStep(wl.B, wl.K, wl.V, wl.topk, wl.n_min, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv,
                           act_dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32)
    Ct = None if inp.C is None else C.dev(inp.C)
    args = (C.dev(inp.logits, wl.dtype), C.dev(inp.root_tok), C.dev(inp.ctx_len), Ct, inp.L_AR,
            C.dev(inp.q, wl.dtype), C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv, inp.scale,
            C.dev(target, wl.dtype))
    step(*args)
    step(*args)   # second call reuses the workspaces
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0
    for k_ in ("n", "parent", "token", "depth", "pos"):
        assert np.array_equal(getattr(step, k_).cpu().numpy(), tree[k_]), k_
    acc = C.oracle_accept(inp, tree, target)
    for k_, wv in zip(("acc_len", "acc_nodes", "acc_tok", "bonus", "argmax"), acc):
        assert np.array_equal(getattr(step, k_).cpu().numpy(), wv), k_
    rows = C.attention_rows(inp, tree, 32)
    want = C.oracle_attention(inp, tree, rows=rows)
    got = step.attn_out.float().cpu().numpy()
    atol, rtol = attn_tol(wl)
    for r in rows:
        assert np.all(np.abs(got[r] - want[r]) <= atol + rtol * np.abs(want[r])), r


def test_long_context_attention_covers_every_head_group_and_m_tile():
    """long_ctx_b4 at full size (4 requests x 32K context, 128 nodes, GQA 32/8):
    rows from every (request, KV head) pair and from each of its four
    128-row M-tiles (nodes 0-31, 32-63, 64-95, 96-127; the M rows pack the
    group's four query heads node by node), each with a different head of the
    group, against the oracle."""
    wl = W["long_ctx_b4"]
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    nodes_per_tile = 128 // wl.g
    rows = []
    for b in range(wl.B):
        nb = int(tree["n"][b])
        for kvh in range(wl.Hkv):
            for m in range((nb * wl.g + 127) // 128):
                i = min(nb - 1, nodes_per_tile * m + (7 * (b + kvh) + 5 * m) % nodes_per_tile)
                rows.append((b, i, kvh * wl.g + (b + kvh + m) % wl.g))
    assert len({(b, h // wl.g) for b, _, h in rows}) == wl.B * wl.Hkv
    _attention_parity(inp, tree, max_rows=0, rows=sorted(set(rows)))


def _fill_host(views, inp, target):
    wl = inp.wl
    src = {"logits": inp.logits, "root_tok": inp.root_tok, "ctx_len": inp.ctx_len, "q": inp.q, "k_tree": inp.k_tree,
           "v_tree": inp.v_tree, "target": target}
    for k_, a in src.items():
        v = views[k_]
        if v.dtype == torch.bfloat16:
            v.view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(v.shape))
        else:
            v.copy_(torch.from_numpy(np.ascontiguousarray(a)).view(v.shape))


@pytest.mark.parametrize("name", ["qwen3_ragged", "paged_ragged", "qwen3_8b_b1"])
def test_host_runner_matches_oracle(name):
    """Steps fed from pinned host blocks through the double-buffered runner:
    two different drafter/target sets in flight at once (same context cache,
    latency table and context lengths, which are the runner's fixed state),
    then a third step that reuses the first slot; every result matches the
    oracle's."""
    import dataclasses
    wl = ALL[name]
    inp0, o0 = C.pick(wl, 0)
    sets = [(inp0, o0)]
    for seed in range(1, 20):   # drafter logits of another seed, without near ties
        other = I.make_step_inputs(wl, seed, with_attention=False)
        cand = dataclasses.replace(inp0, logits=other.logits)
        o = C.oracle_draft(cand)
        if all(g >= C.GAP for g in o["tree"]["gaps"]):
            sets.append((cand, o))
            break
    assert len(sets) == 2
    kv = C.kv_of(inp0)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    step = bn.SpecTreeStep(wl.B, wl.K, wl.V, wl.topk, wl.n_min, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv, act_dtype=dt)
    Ct = None if inp0.C is None else C.dev(inp0.C)
    runner = bn.HostStepRunner(step, kv, Ct, inp0.L_AR, inp0.scale, act_dtype=dt, depth=2)
    wants = []
    for slot, (inp, o) in enumerate(sets):
        tree = o["tree"]
        target = C.target_for(inp, tree)
        _fill_host(runner.inputs(slot), inp, target)
        wants.append((tree, C.oracle_accept(inp, tree, target)))
    order = [0, 1, 0]
    for s in order[:2]:
        assert runner.submit() == s
    got = [runner.collect()]
    assert runner.submit() == 0
    got += [runner.collect(), runner.collect()]
    assert int(step.dev_err.item()) == 0
    assert runner.h2d_bytes >= sum(v.numel() * v.element_size() for v in runner.inputs(0).values())
    for s, g in zip(order, got):
        tree, (acc_len, _, acc_tok, bonus, _) = wants[s]
        assert np.array_equal(g["n"].numpy(), tree["n"])
        assert np.array_equal(g["acc_len"].numpy(), acc_len)
        assert np.array_equal(g["acc_tok"].numpy(), acc_tok)
        assert np.array_equal(g["bonus"].numpy(), bonus)
