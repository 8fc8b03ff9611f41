"""Committing the accepted path to the context KV cache: the CUDA call against
the oracle, bit-exact (pure data movement), contiguous and paged, plus its
device-error cases.  Inputs are the oracle's acceptance results on seeded
workloads, with room added to the cache for the new positions."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402
from .test_gpu_parity import SMALL  # noqa: E402

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


def with_room(inp, extra):
    """Stored-dtype context arrays with `extra` more positions per request:
    contiguous rows grow; paged pools get fresh pages, entered in each block
    table row right after the request's last page (columns added as needed)."""
    wl = inp.wl
    kc, vc, bt = inp.k_ctx, inp.v_ctx, inp.block_table
    if bt is None:
        pad = np.zeros(kc.shape[:2] + (extra,) + kc.shape[3:], kc.dtype)
        return np.concatenate([kc, pad], axis=2), np.concatenate([vc, pad], axis=2), None
    ps = wl.page_size
    per = -(-extra // ps) + 1
    P = kc.shape[0]
    new = np.zeros((wl.B * per,) + kc.shape[1:], kc.dtype)
    bt2 = np.concatenate([bt, np.full((wl.B, per), -1, np.int32)], axis=1)
    for b in range(wl.B):
        used = int((bt[b] >= 0).sum())
        bt2[b, used:used + per] = P + b * per + np.arange(per)
    return np.concatenate([kc, new]), np.concatenate([vc, new]), bt2


def first_child_target(tree, V, dtype):
    """Target rows whose argmax at each node is its first child's token: the
    accepted path runs down first children to a leaf."""
    B, N = tree["parent"].shape
    t = np.zeros((B, N, V), np.float32)
    for b in range(B):
        n = int(tree["n"][b])
        for u in range(n):
            kids = np.nonzero(tree["parent"][b, :n] == u)[0]
            t[b, u, int(tree["token"][b, kids[0]]) if len(kids) else 0] = 1.0
    return I.store(t, dtype)


def run_commit(inp, acc_len, acc_nodes, kc, vc, bt, ctx_len=None, in_place=False):
    wl = inp.wl
    kv = bn.KV(C.dev(kc, wl.dtype), C.dev(vc, wl.dtype), None if bt is None else C.dev(bt))
    ctx = C.dev(inp.ctx_len if ctx_len is None else ctx_len)
    out = ctx if in_place else torch.full_like(ctx, -7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_kv_commit(C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv, C.dev(acc_len),
                         C.dev(acc_nodes), ctx, out, dev_err=err)
    torch.cuda.synchronize()

    def host(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()
    return host(kv.k), host(kv.v), out.cpu().numpy(), int(err.item())


def check(inp, acc_len, acc_nodes, extra, in_place=False):
    kc, vc, bt = with_room(inp, extra)
    want_k, want_v, want_ctx = oracle.kv_commit(inp.k_tree, inp.v_tree, acc_len, acc_nodes, kc, vc, inp.ctx_len,
                                                block_table=bt, page_size=inp.wl.page_size)
    got_k, got_v, got_ctx, err = run_commit(inp, acc_len, acc_nodes, kc, vc, bt, in_place=in_place)
    assert err == 0
    assert np.array_equal(got_ctx, want_ctx)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)


CASES = {**{k: W[k] for k in ("tiny_v1024_f32", "qwen3_8b_b1", "llama31_8b_b16_paged")},
         **{k: SMALL[k] for k in ("qwen3_ragged", "paged_ragged", "mha_d64")}}


@pytest.mark.parametrize("name", list(CASES))
def test_commit_of_the_greedy_path_matches_oracle(name):
    """The path the oracle accepts for the workload's own target rows, and a
    long path (first children down to a leaf)."""
    wl = CASES[name]
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    for target in (C.target_for(inp, tree), first_child_target(tree, wl.V, wl.dtype)):
        acc_len, acc_nodes, *_ = C.oracle_accept(inp, tree, target)
        check(inp, acc_len, acc_nodes, wl.K + 1)
    assert acc_len.max() >= 1   # at least one accepted draft token is committed


def test_commit_in_place_and_full_depth():
    """ctx_out aliasing ctx_len, and the deepest path (acc_len = K) at a
    request whose context ends exactly one path short of the capacity."""
    wl = SMALL["qwen3_ragged"].scaled(name="chain", topk=1, n_min=17, n_max=17)
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    acc_len, acc_nodes, *_ = C.oracle_accept(inp, tree, first_child_target(tree, wl.V, wl.dtype))
    assert (acc_len == wl.K).all()
    check(inp, acc_len, acc_nodes, wl.K + 1, in_place=True)


def test_commit_device_errors_copy_nothing():
    wl = SMALL["paged_ragged"]
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    acc_len, acc_nodes, *_ = C.oracle_accept(inp, tree, first_child_target(tree, wl.V, wl.dtype))
    kc, vc, bt = with_room(inp, wl.K + 1)
    # acc_len beyond K on request 0, a node id beyond n_max on request 1
    bad_len = acc_len.copy()
    bad_len[0] = wl.K + 1
    bad_nodes = acc_nodes.copy()
    bad_nodes[1, 0] = wl.n_max
    k2, v2, ctx2, err = run_commit(inp, bad_len, bad_nodes, kc, vc, bt)
    assert err & bn.DEVERR_N
    assert ctx2[0] == inp.ctx_len[0] and ctx2[1] == inp.ctx_len[1]
    good = list(range(2, wl.B))
    want_k, _, want_ctx = oracle.kv_commit(inp.k_tree[good], inp.v_tree[good], acc_len[good], acc_nodes[good], kc,
                                           vc, inp.ctx_len[good], block_table=bt[good], page_size=wl.page_size)
    assert np.array_equal(k2, want_k) and np.array_equal(ctx2[good], want_ctx)
    # the block table as generated, request 0's context moved to the end of its
    # last page: its next position has no page (BASTION_DEVERR_PAGE, or _CTX
    # when the table has no further column)
    ctx_mod = inp.ctx_len.copy()
    ctx_mod[0] = int((inp.block_table[0] >= 0).sum()) * wl.page_size
    _, _, ctx3, err = run_commit(inp, acc_len, acc_nodes, inp.k_ctx, inp.v_ctx, inp.block_table, ctx_len=ctx_mod)
    assert err & (bn.DEVERR_PAGE | bn.DEVERR_CTX)
    assert ctx3[0] == ctx_mod[0]
    for b in range(1, wl.B):
        assert ctx3[b] in (ctx_mod[b], ctx_mod[b] + acc_len[b] + 1)
    # contiguous cache without room: BASTION_DEVERR_CTX, nothing written
    wl2 = SMALL["qwen3_ragged"]
    inp2, o2 = C.pick(wl2, 0)
    a2, n2, *_ = C.oracle_accept(inp2, o2["tree"], first_child_target(o2["tree"], wl2.V, wl2.dtype))
    k4, _, ctx4, err = run_commit(inp2, a2, n2, inp2.k_ctx, inp2.v_ctx, None)
    assert err & bn.DEVERR_CTX
    assert np.array_equal(ctx4, inp2.ctx_len) and np.array_equal(k4, inp2.k_ctx)


def test_step_then_commit_matches_oracle():
    """The four calls, then the commit fed by the step's own acceptance
    outputs on the device."""
    wl = W["llama31_8b_b16_paged"]
    inp, o = C.pick(wl, 0)
    tree = o["tree"]
    target = first_child_target(tree, wl.V, wl.dtype)
    kc, vc, bt = with_room(inp, wl.K + 1)
    kv = bn.KV(C.dev(kc, wl.dtype), C.dev(vc, wl.dtype), C.dev(bt))
    step = bn.SpecTreeStep(wl.B, wl.K, wl.V, wl.topk, wl.n_min, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv)
    ctx = C.dev(inp.ctx_len)
    kt, vt = C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype)
    step(C.dev(inp.logits, wl.dtype), C.dev(inp.root_tok), ctx, C.dev(inp.C), inp.L_AR, C.dev(inp.q, wl.dtype), kt,
         vt, kv, inp.scale, C.dev(target, wl.dtype))
    bn.bastion_kv_commit(kt, vt, kv, step.acc_len, step.acc_nodes, ctx, ctx, dev_err=step.dev_err)
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0
    acc_len, acc_nodes, *_ = C.oracle_accept(inp, tree, target)
    want_k, want_v, want_ctx = oracle.kv_commit(inp.k_tree, inp.v_tree, acc_len, acc_nodes, kc, vc, inp.ctx_len,
                                                block_table=bt, page_size=wl.page_size)
    assert np.array_equal(ctx.cpu().numpy(), want_ctx)
    assert np.array_equal(kv.k.view(torch.int16).cpu().numpy().view(np.uint16), want_k)
    assert np.array_equal(kv.v.view(torch.int16).cpu().numpy().view(np.uint16), want_v)
