"""Edge cases of the CUDA path: degenerate trees, empty contexts, massive
ties, and the device error word for inputs only the device can check.

Every "bad input" case here is one the kernels check before touching memory
(the access is skipped and a bit is set in the error word); none faults.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402
from .test_gpu_parity import check_stage1, check_tree, run_draft  # noqa: E402

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


def whole_step(inp, tree, target):
    wl = inp.wl
    kv = C.kv_of(inp)
    act = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    step = bn.SpecTreeStep(wl.B, wl.K, wl.V, wl.topk, wl.n_min, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv, act_dtype=act)
    Ct = None if inp.C is None else C.dev(inp.C)
    step(C.dev(inp.logits, wl.dtype), C.dev(inp.root_tok), C.dev(inp.ctx_len), Ct, inp.L_AR, C.dev(inp.q, wl.dtype),
         C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv, inp.scale, C.dev(target, wl.dtype))
    torch.cuda.synchronize()
    return step


def compare_step(inp, tree, target, step):
    wl = inp.wl
    assert int(step.dev_err.item()) == 0
    for k_ in ("n", "parent", "token", "depth", "pos"):
        assert np.array_equal(getattr(step, k_).cpu().numpy(), tree[k_]), k_
    acc = C.oracle_accept(inp, tree, target)
    for k_, wv in zip(("acc_len", "acc_nodes", "acc_tok", "bonus", "argmax"), acc):
        assert np.array_equal(getattr(step, k_).cpu().numpy(), wv), k_
    want = C.oracle_attention(inp, tree)
    got = step.attn_out.float().cpu().numpy()
    atol, rtol = (2e-2, 1e-2) if wl.dtype == "bf16" else (1e-4, 1e-4)
    for b in range(wl.B):
        nb = int(tree["n"][b])
        assert np.all(np.abs(got[b, :nb] - want[b, :nb]) <= atol + rtol * np.abs(want[b, :nb]))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_root_only_tree(dtype):
    """n_min = n_max = 1: the tree is the root; attention sees context + itself;
    acceptance returns length 0 and the root's argmax as bonus."""
    wl = W["qwen3_8b_b1"].scaled(name="root_only", B=3, V=3000, K=4, n_min=1, n_max=1, L=150, dtype=dtype)
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    assert (tree["n"] == 1).all()
    target = C.target_for(inp, tree)
    step = whole_step(inp, tree, target)
    compare_step(inp, tree, target, step)
    assert (step.acc_len.cpu().numpy() == 0).all()


def test_empty_context():
    """ctx_len = 0: the nodes attend to their tree path only."""
    wl = W["qwen3_8b_b1"].scaled(name="empty_ctx", B=2, V=4096, K=5, n_min=20, n_max=20, L=64)
    inp, o = C.pick(wl, 0)
    inp.ctx_len[:] = 0
    tree = o["tree"]
    tree = dict(tree)
    tree["pos"] = tree["depth"].copy()
    tree["pos"][tree["depth"] < 0] = -1
    target = C.target_for(inp, tree)
    step = whole_step(inp, tree, target)
    compare_step(inp, tree, target, step)


def test_constant_logits_take_the_tie_path():
    """Every logit equal: top-k is ids 0..k-1 (lowest ids win ties) through the
    exact-selection fallback, and the tree breaks every equal-rho tie by token
    id then parent index, identically to the oracle."""
    wl = W["qwen3_8b_b1"].scaled(name="constant", B=2, V=50000, K=4, topk=5, n_min=40, n_max=40, L=16)
    inp = I.make_step_inputs(wl, 0, with_attention=False)
    inp.logits[...] = I.to_bf16_bits(np.full(1, 1.5, np.float32))[0]
    o = C.oracle_draft(inp)
    s1, tree = run_draft(inp)
    check_stage1(wl, s1, o)
    assert (s1["ids"][..., :5] == np.arange(5)).all()
    check_tree(tree, o["tree"])


@pytest.mark.parametrize("name", ["bf16_v20000", "f32_v1001"])
def test_topk_streams_more_rows_than_clusters(name):
    """More drafter rows than clusters fit on the device at once: each cluster
    streams several rows through its staging buffer and rank 0's two inbox
    buffers.  Every row is checked against the oracle."""
    wl = {"bf16_v20000": W["qwen3_8b_b1"].scaled(name="rows_bf16", B=80, K=16, V=20000, topk=8),
          "f32_v1001": W["tiny_v1024_f32"].scaled(name="rows_f32", B=100, K=8, V=1001, topk=7)}[name]
    inp = I.make_step_inputs(wl, 3, with_attention=False)
    R = wl.rows
    x = I.as_f32(inp.logits, wl.dtype).reshape(R, wl.V)
    want = dict(zip(("ids", "lg", "q", "lse"), oracle.topk_softmax(x, wl.topk)))
    got = dict(ids=torch.empty(R, wl.topk, dtype=torch.int32, device="cuda"),
               lg=torch.empty(R, wl.topk, dtype=torch.float32, device="cuda"),
               q=torch.empty(R, wl.topk, dtype=torch.float32, device="cuda"),
               lse=torch.empty(R, dtype=torch.float64, device="cuda"))
    bn.bastion_topk_softmax(C.dev(inp.logits, wl.dtype).reshape(R, wl.V), wl.topk, got["ids"], got["lg"], got["q"],
                            got["lse"])
    torch.cuda.synchronize()
    check_stage1(wl, {k_: v.cpu().numpy() for k_, v in got.items()}, want)


def test_chain_k1():
    """k = 1: the tree is the greedy top-1 chain."""
    wl = W["controller_sweep_peaked"].scaled(name="chain", B=2, V=9000, topk=1, n_min=1, n_max=40, L=100)
    inp, o = C.pick(wl, 0)
    s1, tree = run_draft(inp)
    check_tree(tree, o["tree"])
    for b in range(wl.B):
        nb = int(tree["n"][b])
        assert (tree["parent"][b, 1:nb] == np.arange(nb - 1)).all()


# --------------------------------------------------------------------------
# device error word
# --------------------------------------------------------------------------


def _tree_bufs(B, N):
    t = {k: torch.empty(B, N, dtype=torch.int32, device="cuda") for k in ("parent", "token", "depth", "pos")}
    t["n"] = torch.empty(B, dtype=torch.int32, device="cuda")
    t["rho"] = torch.empty(B, N, dtype=torch.float32, device="cuda")
    t["mask"] = torch.empty(B, N, (N + 63) // 64, dtype=torch.int64, device="cuda")
    t["ahat"] = torch.empty(B, dtype=torch.float32, device="cuda")
    t["S"] = torch.empty(B, dtype=torch.float32, device="cuda")
    return t


def test_token_out_of_range_sets_error_bit():
    B, K, k, N, V = 1, 3, 2, 6, 100
    ids = torch.tensor([[[1, 2], [3, 150], [5, 6]]], dtype=torch.int32, device="cuda")   # 150 >= V
    lg = torch.tensor([[[2.0, 1.0], [2.0, 1.0], [2.0, 1.0]]], dtype=torch.float32, device="cuda")
    lse = torch.full((B, K), 3.0, dtype=torch.float64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = _tree_bufs(B, N)
    bn.bastion_tree_build(ids, lg, lse, V, torch.zeros(B, dtype=torch.int32, device="cuda"),
                          torch.zeros(B, dtype=torch.int32, device="cuda"), N, N, None, 1.0, t["n"], t["parent"],
                          t["token"], t["depth"], t["pos"], t["rho"], t["mask"], t["ahat"], t["S"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & bn.DEVERR_TOKEN
    assert int(t["n"].item()) == N          # the kernel still completed


def _attn_case(paged):
    base = W["llama31_8b_b16_paged"] if paged else W["qwen3_8b_b1"]
    wl = base.scaled(name="err", B=2, V=2048, K=3, topk=3, n_min=8, n_max=8, L=100, L_min=40 if paged else 0)
    inp, o = C.pick(wl, 0)
    return wl, inp, o["tree"]


def _run_attn(wl, inp, tree, n, ctx_len, block_table=None):
    kv = C.kv_of(inp)
    if block_table is not None:
        kv = bn.KV(kv.k, kv.v, block_table)
    out = torch.zeros(wl.B, wl.n_max, wl.Hq, wl.d, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(max(1, bn.bastion_tree_attn_workspace_size(wl.B, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv)),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_tree_attn(C.dev(inp.q, "bf16"), C.dev(inp.k_tree, "bf16"), C.dev(inp.v_tree, "bf16"), kv, ctx_len,
                         C.dev(tree["mask"].view(np.int64)), n, out, inp.scale, ws=ws, dev_err=err)
    torch.cuda.synchronize()
    return int(err.item())


def test_attention_error_bits():
    wl, inp, tree = _attn_case(False)
    n_ok, ctx_ok = C.dev(tree["n"]), C.dev(inp.ctx_len)
    assert _run_attn(wl, inp, tree, n_ok, ctx_ok) == 0
    bad_n = n_ok.clone()
    bad_n[1] = 0
    assert _run_attn(wl, inp, tree, bad_n, ctx_ok) & bn.DEVERR_N
    bad_n[1] = wl.n_max + 3
    assert _run_attn(wl, inp, tree, bad_n, ctx_ok) & bn.DEVERR_N
    bad_ctx = ctx_ok.clone()
    bad_ctx[0] = inp.k_ctx.shape[2] + 50      # beyond the contiguous cache
    assert _run_attn(wl, inp, tree, n_ok, bad_ctx) & bn.DEVERR_CTX


def test_paged_attention_bad_page_sets_error_bit():
    wl, inp, tree = _attn_case(True)
    bt = C.dev(inp.block_table)
    ctx = C.dev(inp.ctx_len)
    assert _run_attn(wl, inp, tree, C.dev(tree["n"]), ctx, bt) == 0
    bad = bt.clone()
    bad[0, 0] = inp.k_ctx.shape[0] + 7        # page id past the pool
    assert _run_attn(wl, inp, tree, C.dev(tree["n"]), ctx, bad) & bn.DEVERR_PAGE


def test_accept_invalid_n_sets_error_bit_and_fills_minus_one():
    B, N, V, K = 2, 8, 500, 4
    target = torch.randn(B, N, V, device="cuda").to(torch.bfloat16)
    n = torch.tensor([3, N + 1], dtype=torch.int32, device="cuda")
    parent = torch.tensor([[-1, 0, 0, -1, -1, -1, -1, -1]] * 2, dtype=torch.int32, device="cuda")
    token = torch.tensor([[7, 1, 2, -1, -1, -1, -1, -1]] * 2, dtype=torch.int32, device="cuda")
    out = {k: torch.zeros(*s, dtype=torch.int32, device="cuda")
           for k, s in (("len", (B,)), ("nodes", (B, K + 1)), ("tok", (B, K + 1)), ("bonus", (B,)), ("am", (B, N)))}
    ws = torch.zeros(bn.bastion_accept_workspace_size(B, N), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_accept(target, n, parent, token, K, out["len"], out["nodes"], out["tok"], out["bonus"], ws,
                      argmax_out=out["am"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & bn.DEVERR_N
    assert int(out["len"][1].item()) == -1 and (out["nodes"][1] == -1).all() and (out["am"][1] == -1).all()
    # request 0 is unaffected
    want = oracle.accept(target[:1].float().cpu().numpy(), np.array([3]), parent[:1].cpu().numpy(),
                         token[:1].cpu().numpy(), K)
    assert int(out["len"][0].item()) == int(want[0][0])
    assert int(out["bonus"][0].item()) == int(want[3][0])


# --------------------------------------------------------------------------
# signed zeros: -0.0 and +0.0 are equal values, so ties between them go to
# the lower id, as in the oracle (a float comparison, not a bit comparison)
# --------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_accept_argmax_ties_between_signed_zeros(dtype):
    """Rows whose maximum is zero, held as -0.0 and +0.0 at different ids: in
    different CTAs (chunks), in different threads of one CTA, in the same
    16-byte vector, and with +0.0 first.  The argmax is the lowest id of
    either sign, as np.argmax gives."""
    B, N, V, K = 1, 6, 151936, 4
    rows = np.full((B, N, V), -1.0, np.float32)
    zeros = {0: [(100, -0.0), (100000, 0.0)],     # chunk 0 vs a later chunk
             1: [(50, 0.0), (60, -0.0)],          # +0.0 first
             2: [(8, -0.0), (3000, 0.0)],         # two threads of one CTA
             3: [(3, -0.0), (2, 0.0)],            # one 16-byte vector, +0.0 lower
             4: [(40000, -0.0), (30000, -0.0), (151935, 0.0)],
             5: [(7, 0.0)]}
    for i, zs in zeros.items():
        for j, z in zs:
            rows[0, i, j] = z
    stored = I.store(rows, dtype)
    target = C.dev(stored, dtype)
    n = torch.tensor([N], dtype=torch.int32, device="cuda")
    parent_h = np.array([[-1, 0, 0, 1, 1, 2]], np.int32)
    token_h = np.array([[5, 100, 50, 8, 2, 3]], np.int32)
    parent, token = C.dev(parent_h), C.dev(token_h)
    out = {k: torch.full(s, -7, dtype=torch.int32, device="cuda")
           for k, s in (("len", (B,)), ("nodes", (B, K + 1)), ("tok", (B, K + 1)), ("bonus", (B,)), ("am", (B, N)))}
    ws = torch.zeros(bn.bastion_accept_workspace_size(B, N), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_accept(target, n, parent, token, K, out["len"], out["nodes"], out["tok"], out["bonus"], ws,
                      argmax_out=out["am"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.accept(C.fview(stored, dtype), np.array([N]), parent_h, token_h, K)
    assert list(want[4][0]) == [100, 50, 8, 2, 30000, 7]
    for k_, wv in zip(("len", "nodes", "tok", "bonus", "am"), want):
        assert np.array_equal(out[k_].cpu().numpy(), wv), k_


def test_topk_ties_between_signed_zeros():
    """Every logit zero, even ids -0.0 and odd ids +0.0: all are equal, so the
    top-k is ids 0..k-1 (through the exact-selection path for massive ties),
    the logits come back with their own signs, and the tree matches the
    oracle's."""
    wl = W["qwen3_8b_b1"].scaled(name="signed_zero", B=2, V=50000, K=4, topk=5, n_min=30, n_max=30, L=16)
    inp = I.make_step_inputs(wl, 0, with_attention=False)
    z = np.zeros(wl.V, np.float32)
    z[0::2] = -0.0
    inp.logits[...] = I.to_bf16_bits(z)
    o = C.oracle_draft(inp)
    s1, tree = run_draft(inp)
    check_stage1(wl, s1, o)
    assert (s1["ids"][..., :5] == np.arange(5)).all()
    assert np.array_equal(np.signbit(s1["lg"].reshape(-1, 5)), np.signbit(o["lg"]))
    check_tree(tree, o["tree"])


@pytest.mark.parametrize("dtype,V", [("f32", 262144), ("bf16", 262144), ("f32", 262143), ("bf16", 262140)])
def test_topk_at_the_largest_vocabulary(dtype, V):
    """V = 262144 and k = 32: every CTA of a row's cluster ranks its chunk
    and the rank-0 merge takes the best 32 of them.  Row 0 is random (a heavy
    upper tail), row 1 all equal (the exact-selection fallback in every
    chunk), row 2 random with its maximum in the last element; odd V takes
    the unaligned path."""
    k, R = 32, 3
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((R, V)) * 3.0).astype(np.float32)
    x[1] = 0.25
    x[2, -1] = x[2].max() + 4.0
    bits = I.store(x, dtype)
    x = I.as_f32(bits, dtype)
    want = dict(zip(("ids", "lg", "q", "lse"), oracle.topk_softmax(x, k)))
    got = dict(ids=torch.empty(R, k, dtype=torch.int32, device="cuda"),
               lg=torch.empty(R, k, dtype=torch.float32, device="cuda"),
               q=torch.empty(R, k, dtype=torch.float32, device="cuda"),
               lse=torch.empty(R, dtype=torch.float64, device="cuda"))
    bn.bastion_topk_softmax(C.dev(bits, dtype), k, got["ids"], got["lg"], got["q"], got["lse"])
    torch.cuda.synchronize()
    wl = W["qwen3_8b_b1"].scaled(name="max_vocab", B=R, K=1, V=V, topk=k)
    check_stage1(wl, {k_: v.cpu().numpy() for k_, v in got.items()}, want)
    assert (got["ids"][1].cpu().numpy() == np.arange(k)).all()
    assert int(got["ids"][2, 0]) == V - 1


def test_prepared_step_launches_on_call_and_matches_the_oracle():
    """SpecTreeStep.prepare checks and marshals the four calls once and
    launches nothing; each call of the prepared step then runs the whole step
    on the inputs' current contents (here: the controller's S(N) stop, bf16)."""
    wl = W["controller_sweep_flat"].scaled(name="prepared", B=3, V=12288, n_min=2, n_max=48, L=200)
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    target = C.target_for(inp, tree)
    kv = C.kv_of(inp)
    step = bn.SpecTreeStep(wl.B, wl.K, wl.V, wl.topk, wl.n_min, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv,
                           act_dtype=torch.bfloat16)
    Ct = None if inp.C is None else C.dev(inp.C)
    args = (C.dev(inp.logits, wl.dtype), C.dev(inp.root_tok), C.dev(inp.ctx_len), Ct, inp.L_AR,
            C.dev(inp.q, wl.dtype), C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv, inp.scale,
            C.dev(target, wl.dtype))
    step.result.fill_(-7)
    prepared = step.prepare(*args)
    torch.cuda.synchronize()
    assert (step.result.cpu().numpy() == -7).all()    # nothing ran yet
    for _ in range(2):                                # repeatable on the same workspaces
        step.result.fill_(-7)
        prepared()
        torch.cuda.synchronize()
        compare_step(inp, tree, target, step)
    with pytest.raises(bn.BastionError):              # checks still run when preparing
        step.prepare(*args[:5], args[5].float(), *args[6:])
