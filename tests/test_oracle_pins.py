"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against a closed form, a library routine, a brute
force enumeration on tiny inputs, an invariant the BASTION explainer pages
state, or the pages' own worked example (tests/golden/).  The cases are chosen
so that a plausible slip (root left out of A_hat, a child taken from the wrong
position, a reversed tie-break, a transposed operand) fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from tree_speculative_decoding_bastion_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# stage 1: marginals and top-k
# --------------------------------------------------------------------------


def test_marginals_closed_form():
    # exp(0) : exp(ln 2) : exp(ln 3) = 1 : 2 : 3, normaliser 6
    q, lse = oracle.marginals(np.array([0.0, math.log(2.0), math.log(3.0)]))
    np.testing.assert_allclose(q, [1 / 6, 2 / 6, 3 / 6], rtol=1e-14)
    assert abs(lse - math.log(6.0)) < 1e-14


def test_marginals_match_scipy_and_sum_to_one():
    rng = np.random.default_rng(11)
    for V in (1, 7, 1000, 4097):
        x = (rng.standard_normal(V) * 3 + 20).astype(np.float32)
        q, lse = oracle.marginals(x)
        np.testing.assert_allclose(q, scipy.special.softmax(x.astype(np.float64)), rtol=1e-12, atol=0)
        assert abs(lse - scipy.special.logsumexp(x.astype(np.float64))) < 1e-12
        assert abs(q.sum() - 1.0) < 1e-12


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(20):
        V = int(rng.integers(1, 60))
        k = int(rng.integers(1, min(V, 32) + 1))
        # integer-valued logits give many exact ties
        x = rng.integers(-3, 4, size=(3, V)).astype(np.float32)
        ids, lg, q, lse = oracle.topk_softmax(x, k)
        for r in range(3):
            want = sorted(range(V), key=lambda v: (-float(x[r, v]), v))[:k]
            assert ids[r].tolist() == want
            assert lg[r].tolist() == [float(x[r, v]) for v in want]
            qs = scipy.special.softmax(x[r].astype(np.float64))
            np.testing.assert_allclose(q[r], qs[want], rtol=1e-12)


def test_topk_lowest_id_first_on_tie():
    x = np.array([[1.0, 5.0, 5.0, 2.0, 5.0]], dtype=np.float32)
    ids, lg, q, lse = oracle.topk_softmax(x, 4)
    assert ids[0].tolist() == [1, 2, 4, 3]


# --------------------------------------------------------------------------
# stage 2: best-first tree and controller
# --------------------------------------------------------------------------


def _stage1(logits_bkv):
    B, K, V = logits_bkv.shape
    return logits_bkv.reshape(B * K, V)


def _tree_from_logits(x, k, n_max, n_min=None, C=None, L_AR=1.0, root_tok=None, ctx_len=None, tau=0.0):
    """x [B, K, V] -> (trees, ids, lg, lse) through the oracle's stages 1-2."""
    B, K, V = x.shape
    ids, lg, q, lse = oracle.topk_softmax(x.reshape(B * K, V), k)
    ids, lg, lse = ids.reshape(B, K, k), lg.reshape(B, K, k), lse.reshape(B, K)
    root_tok = np.zeros(B, np.int32) if root_tok is None else root_tok
    ctx_len = np.zeros(B, np.int32) if ctx_len is None else ctx_len
    trees = oracle.tree_build(ids, lg, lse, root_tok, ctx_len,
                              n_max if n_min is None else n_min, n_max, C, L_AR, tau)
    return trees, ids, lg, lse


def test_toy_example_from_the_page():
    with open(os.path.join(GOLDEN, "toy_katze_hund.json")) as f:
        g = json.load(f)
    qv = np.array(g["q"], dtype=np.float64)
    x = np.log(qv).astype(np.float32)[None]          # logits whose softmax is q
    n_max = g["n_max"]
    trees, ids, lg, lse = _tree_from_logits(x, 2, n_max, root_tok=np.array([g["root_token"]], np.int32))
    t = trees[0]
    e = g["expected"]
    assert t.n == n_max
    assert t.parent.tolist() == e["parent"]
    assert t.token.tolist() == e["token"]
    assert t.depth.tolist() == e["depth"]
    np.testing.assert_allclose(t.rho, e["rho"], rtol=1e-6)
    np.testing.assert_allclose(np.cumsum(t.rho), e["ahat_by_n"], rtol=1e-6)
    np.testing.assert_allclose(t.S_curve, e["ahat_by_n"], rtol=1e-6)   # C = 1, L_AR = 1
    d1 = {int(t.token[i]): t.rho[i] for i in range(t.n) if t.depth[i] == 1}
    assert abs(d1[g["vocab"]["Katze"]] - g["depth1_rho"]["Katze"]) < 1e-6
    assert abs(d1[g["vocab"]["Hund"]] - g["depth1_rho"]["Hund"]) < 1e-6


def _trie(K, k):
    """All trie nodes as tuples of child ranks, BFS (index) order."""
    nodes = [()]
    frontier = [()]
    for _ in range(K):
        frontier = [p + (j,) for p in frontier for j in range(k)]
        nodes += frontier
    return nodes


def _rho_bruteforce(x_bkv, b, path_ranks, ids):
    """rho of a trie node from an independent softmax (scipy), by definition."""
    r = 1.0
    for d, j in enumerate(path_ranks):
        qs = scipy.special.softmax(x_bkv[b, d].astype(np.float64))
        r *= qs[int(ids[b, d, j])]
    return r


@pytest.mark.parametrize("K,k,V,seed", [(2, 2, 6, 0), (3, 2, 5, 1), (2, 3, 7, 2), (3, 3, 9, 3)])
def test_best_first_is_optimal_bruteforce(K, k, V, seed):
    """max over prefix-closed trees of size n of sum rho == oracle A_hat(n)."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((1, K, V)) * 1.5).astype(np.float32)
    nodes = _trie(K, k)
    n_max = min(8, len(nodes))
    trees, ids, lg, lse = _tree_from_logits(x, k, n_max)
    t = trees[0]
    rho = [_rho_bruteforce(x, 0, p, ids) for p in nodes]
    index = {p: i for i, p in enumerate(nodes)}
    best = [0.0] * (n_max + 1)

    def grow(chosen, total, last):
        n = len(chosen)
        best[n] = max(best[n], total)
        if n == n_max:
            return
        for j in range(last + 1, len(nodes)):
            p = nodes[j]
            if p[:-1] in chosen:
                chosen.add(p)
                grow(chosen, total + rho[j], j)
                chosen.remove(p)

    grow({()}, rho[0], 0)
    ahat = np.cumsum(t.rho[: t.n])
    for n in range(1, n_max + 1):
        assert abs(ahat[n - 1] - best[n]) < 1e-9, (n, ahat[n - 1], best[n])


@pytest.mark.parametrize("seed", range(4))
def test_tree_is_top_n_of_trie_and_rho_is_path_product(seed):
    rng = np.random.default_rng(100 + seed)
    K, k, V, B = 3, 3, 11, 2
    x = (rng.standard_normal((B, K, V)) * 2).astype(np.float32)
    n_max = 20
    trees, ids, lg, lse = _tree_from_logits(x, k, n_max, ctx_len=np.array([5, 9], np.int32))
    nodes = _trie(K, k)
    for b, t in enumerate(trees):
        rho_all = sorted(((_rho_bruteforce(x, b, p, ids), p) for p in nodes), reverse=True)
        top = {p for _, p in rho_all[:n_max]}
        # reconstruct each tree node's rank path from parent/token
        got = set()
        for i in range(t.n):
            path = oracle.path_to_root(t.parent, i)[1:]
            ranks = tuple(int(np.where(ids[b, d] == t.token[j])[0][0]) for d, j in enumerate(path))
            got.add(ranks)
            assert abs(t.rho[i] - _rho_bruteforce(x, b, ranks, ids)) < 1e-12 * max(1.0, t.rho[i]) + 1e-15
            assert t.depth[i] == len(path)
            assert t.pos[i] == [5, 9][b] + len(path)
        assert got == top


@pytest.mark.parametrize("seed", range(3))
def test_ahat_nondecreasing_concave(seed):
    wl = inputs.WORKLOADS["tiny_v1024_f32"].scaled(n_max=64, n_min=64)
    inp = inputs.make_step_inputs(wl, seed, with_attention=False)
    x = inputs.as_f32(inp.logits, wl.dtype)
    trees, *_ = _tree_from_logits(x, wl.topk, wl.n_max)
    for t in trees:
        r = t.rho[: t.n]
        assert np.all(np.diff(r) <= 1e-15)          # pop rho nonincreasing
        a = np.cumsum(r)
        assert np.all(np.diff(a) >= 0)              # A_hat nondecreasing
        assert np.all(np.diff(a, 2) <= 1e-15)       # and concave


def test_k1_chain_closed_form():
    rng = np.random.default_rng(3)
    K, V = 6, 40
    x = (rng.standard_normal((1, K, V)) * 2).astype(np.float32)
    trees, ids, lg, lse = _tree_from_logits(x, 1, 50)
    t = trees[0]
    assert t.n == K + 1                       # the whole chain, then exhausted
    assert t.parent[: t.n].tolist() == [-1] + list(range(K))
    qtop = [scipy.special.softmax(x[0, d].astype(np.float64)).max() for d in range(K)]
    want = 1.0 + sum(np.prod(qtop[: d + 1]) for d in range(K))
    assert abs(t.ahat - want) < 1e-12
    assert t.token[1 : t.n].tolist() == [int(np.argmax(x[0, d])) for d in range(K)]


def test_mask_is_ancestor_or_self():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((1, 4, 30)) * 1.0).astype(np.float32)
    trees, *_ = _tree_from_logits(x, 4, 100)
    t = trees[0]
    assert t.n == 100 and t.mask.shape == (100, 2)
    for i in range(t.n):
        anc = set(oracle.path_to_root(t.parent, i))
        for j in range(t.n):
            bit = (int(t.mask[i, j // 64]) >> (j % 64)) & 1
            assert bit == (j in anc)
        assert t.parent[i] < i                     # topological pop order


def _controller_case(seed, n_min, n_max, regime):
    wl = inputs.WORKLOADS["controller_sweep_" + regime].scaled(V=2048, n_min=n_min, n_max=n_max, B=2)
    inp = inputs.make_step_inputs(wl, seed, with_attention=False)
    x = inputs.as_f32(inp.logits, wl.dtype)
    return wl, inp, x


@pytest.mark.parametrize("regime", ["peaked", "flat"])
@pytest.mark.parametrize("seed", range(3))
def test_controller_first_drop_is_argmax_of_S(regime, seed):
    """S(n) = A_hat(n) L_AR / C(n) recomputed from the table; the first drop
    after n_min equals argmax over [n_min, n_max] (A_hat concave, C affine-
    convex, so S is unimodal)."""
    n_min, n_max = 1, 96
    wl, inp, x = _controller_case(seed, n_min, n_max, regime)
    C, L_AR = inp.C, inp.L_AR
    fixed, *_ = _tree_from_logits(x, wl.topk, n_max)
    ctrl, *_ = _tree_from_logits(x, wl.topk, n_max, n_min=n_min, C=C, L_AR=L_AR)
    # the tree under the controller is a prefix of the fixed-budget pop order
    for tf, tc in zip(fixed, ctrl):
        assert tc.parent[: tc.n].tolist() == tf.parent[: tc.n].tolist()
        assert tc.token[: tc.n].tolist() == tf.token[: tc.n].tolist()
        a = np.cumsum(tf.rho[: tf.n])
        S = np.array([a[n - 1] * L_AR / float(C[n]) for n in range(1, tf.n + 1)])
        np.testing.assert_allclose(tc.S_curve[: tc.n], S[: tc.n], rtol=1e-12)
        assert abs(tc.S - S[tc.n - 1]) < 1e-12 * S[tc.n - 1]
        lo = n_min - 1
        assert tc.n == lo + 1 + int(np.argmax(S[lo:]))


def test_controller_respects_n_min():
    wl, inp, x = _controller_case(0, 1, 64, "flat")
    C = inp.C.copy()
    # C(n+1)/C(n) = 3 > A_hat(n+1)/A_hat(n) (at most 2, as rho <= 1 <= A_hat):
    # every added node lowers S
    C[1:] = C[1] * np.float32(3.0) ** np.arange(64, dtype=np.float32)
    t1, *_ = _tree_from_logits(x, wl.topk, 64, n_min=1, C=C, L_AR=inp.L_AR)
    t5, *_ = _tree_from_logits(x, wl.topk, 64, n_min=5, C=C, L_AR=inp.L_AR)
    assert all(t.n == 1 for t in t1)
    assert all(t.n == 5 for t in t5)


# --------------------------------------------------------------------------
# stage 3: tree attention
# --------------------------------------------------------------------------


def _sdpa(qv, keys, values, scale):
    qt = torch.tensor(qv, dtype=torch.float64).view(1, 1, 1, -1)
    kt = torch.tensor(keys, dtype=torch.float64).view(1, 1, keys.shape[0], -1)
    vt = torch.tensor(values, dtype=torch.float64).view(1, 1, values.shape[0], -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale).view(-1).numpy()


def _small_attention_case(seed, layout="contiguous"):
    base = inputs.WORKLOADS["llama31_8b_b16_paged" if layout == "paged" else "qwen3_8b_b1"]
    wl = base.scaled(B=2, K=3, V=64, topk=3, n_min=10, n_max=10, controller=False, Hq=4, Hkv=2,
                     d=16, L=40, L_min=17 if layout == "paged" else 0, page_size=16)
    inp = inputs.make_step_inputs(wl, seed)
    x = inputs.as_f32(inp.logits, wl.dtype)
    trees, *_ = _tree_from_logits(x, wl.topk, wl.n_max, ctx_len=inp.ctx_len)
    T = oracle.stack_trees(trees)
    f = lambda a: inputs.as_f32(a, wl.dtype)
    out = oracle.tree_attention(f(inp.q), f(inp.k_tree), f(inp.v_tree), f(inp.k_ctx), f(inp.v_ctx),
                                inp.ctx_len, T["parent"], T["n"], wl.Hkv, inp.scale,
                                block_table=inp.block_table, page_size=wl.page_size)
    return wl, inp, T, out, f


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_tree_attention_matches_sdpa_on_explicit_path(layout):
    wl, inp, T, out, f = _small_attention_case(1, layout)
    q, kt, vt, kc, vc = (f(a) for a in (inp.q, inp.k_tree, inp.v_tree, inp.k_ctx, inp.v_ctx))
    g = wl.Hq // wl.Hkv
    for b in range(wl.B):
        L = int(inp.ctx_len[b])
        for i in range(int(T["n"][b])):
            # walk the parents explicitly (independent of the oracle's helper)
            path, j = [], i
            while j != -1:
                path.insert(0, j)
                j = int(T["parent"][b, j])
            for h in range(wl.Hq):
                kvh = h // g
                if inp.block_table is None:
                    ck, cv = kc[b, kvh, :L], vc[b, kvh, :L]
                else:
                    ck = np.stack([kc[inp.block_table[b, t // 16], kvh, t % 16] for t in range(L)])
                    cv = np.stack([vc[inp.block_table[b, t // 16], kvh, t % 16] for t in range(L)])
                keys = np.concatenate([ck, kt[b, path, kvh]])
                vals = np.concatenate([cv, vt[b, path, kvh]])
                want = _sdpa(q[b, i, h], keys, vals, inp.scale)
                np.testing.assert_allclose(out[b, i, h], want, rtol=1e-10, atol=1e-12)
        assert np.all(np.isnan(out[b, int(T["n"][b]):]))


def test_chain_tree_is_causal_decoding_attention():
    """k = 1 makes the tree a chain: node i sees the context and chain[0..i],
    which is causal attention over the sequence context ++ chain."""
    rng = np.random.default_rng(4)
    L, n, d = 12, 5, 8
    kc, vc = rng.standard_normal((1, 1, L, d)), rng.standard_normal((1, 1, L, d))
    kt, vt = rng.standard_normal((1, n, 1, d)), rng.standard_normal((1, n, 1, d))
    q = rng.standard_normal((1, n, 1, d))
    parent = np.array([[-1, 0, 1, 2, 3]])
    out = oracle.tree_attention(q, kt, vt, kc, vc, np.array([L]), parent, np.array([n]), 1, 0.3)
    seq_k = torch.tensor(np.concatenate([kc[0, 0], kt[0, :, 0]]))[None, None]
    seq_v = torch.tensor(np.concatenate([vc[0, 0], vt[0, :, 0]]))[None, None]
    qq = torch.tensor(q[0, :, 0])[None, None]
    allowed = torch.zeros(n, L + n, dtype=torch.bool)
    for i in range(n):
        allowed[i, : L + i + 1] = True
    want = torch.nn.functional.scaled_dot_product_attention(qq, seq_k, seq_v, attn_mask=allowed, scale=0.3)
    np.testing.assert_allclose(out[0, :, 0], want[0, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    d = 6
    keys = np.tile(rng.standard_normal(d), (9, 1))       # identical keys: uniform weights
    vals = rng.standard_normal((9, d))
    np.testing.assert_allclose(oracle.attend(rng.standard_normal(d), keys, vals, 0.7), vals.mean(0), rtol=1e-12)
    one = oracle.attend(rng.standard_normal(d), keys[:1], vals[:1], 0.7)   # single key: its value
    np.testing.assert_allclose(one, vals[0], rtol=1e-14)


# --------------------------------------------------------------------------
# stage 4: acceptance
# --------------------------------------------------------------------------


def _accept_bruteforce(target, n, parent, token):
    """Longest root path whose every token equals the target argmax at its
    parent (found by checking all nodes, not by walking)."""
    amax = [int(np.argmax(target[i])) for i in range(n)]
    best_len, best_node = 0, 0
    for v in range(n):
        path = []
        j = v
        while j != -1:
            path.insert(0, j)
            j = int(parent[j])
        ok = all(amax[path[s - 1]] == int(token[path[s]]) for s in range(1, len(path)))
        if ok and len(path) - 1 > best_len:
            best_len, best_node = len(path) - 1, v
    return best_len, best_node, amax[best_node]


@pytest.mark.parametrize("seed", range(6))
def test_accept_matches_bruteforce(seed):
    rng = np.random.default_rng(seed)
    K, k, V, n_max, B = 4, 3, 12, 30, 3
    x = (rng.standard_normal((B, K, V)) * 2).astype(np.float32)
    trees, *_ = _tree_from_logits(x, k, n_max)
    T = oracle.stack_trees(trees)
    # target: drafter row of the child position plus noise (often agrees)
    target = np.zeros((B, n_max, V), np.float32)
    for b in range(B):
        for i in range(T["n"][b]):
            target[b, i] = x[b, min(T["depth"][b, i] + 1, K) - 1] + rng.standard_normal(V) * 0.7
    acc_len, acc_nodes, acc_tok, bonus, amax = oracle.accept(target, T["n"], T["parent"], T["token"], K)
    for b in range(B):
        L, node, bon = _accept_bruteforce(target[b], int(T["n"][b]), T["parent"][b], T["token"][b])
        assert acc_len[b] == L and acc_nodes[b, L] == node and bonus[b] == bon
        assert acc_tok[b, L] == bon and (acc_tok[b, L + 1:] == -1).all()
        assert acc_len[b] <= min(K, T["depth"][b].max())
        assert [int(T["token"][b, v]) for v in acc_nodes[b, 1 : L + 1]] == acc_tok[b, :L].tolist()


def test_accept_chain_is_longest_matching_prefix_and_ties_take_lowest_id():
    n, V = 5, 6
    parent = np.array([[-1, 0, 1, 2, 3]])
    token = np.array([[9, 2, 4, 1, 5]])
    target = np.zeros((1, n, V), np.float32)
    target[0, 0, 2] = 1.0          # agrees with node 1 (token 2)
    target[0, 1, 4] = 1.0          # agrees with node 2 (token 4)
    target[0, 2, 3] = 1.0          # disagrees with node 3 (token 1): stop, bonus 3
    target[0, 2, 0] = 1.0          # tie 0 vs 3 -> lowest id 0 is the argmax
    acc_len, acc_nodes, acc_tok, bonus, amax = oracle.accept(target, np.array([n]), parent, token, 4)
    assert acc_len[0] == 2 and acc_nodes[0].tolist() == [0, 1, 2, -1, -1]
    assert bonus[0] == 0 and acc_tok[0].tolist() == [2, 4, 0, -1, -1]


# ---------------------------------------------------------------- KV commit


def _with_room(inp, wl, extra):
    """Context arrays with `extra` more positions of capacity per request
    (contiguous: longer rows; paged: fresh pages appended to every block-table
    row)."""
    f = lambda a: inputs.as_f32(a, wl.dtype).astype(np.float64)
    kc, vc = f(inp.k_ctx), f(inp.v_ctx)
    if inp.block_table is None:
        pad = np.zeros(kc.shape[:2] + (extra,) + kc.shape[3:])
        return np.concatenate([kc, pad], axis=2), np.concatenate([vc, pad], axis=2), None
    P = kc.shape[0]
    per = -(-extra // wl.page_size)
    new = np.zeros((wl.B * per,) + kc.shape[1:])
    bt = np.concatenate([inp.block_table, P + np.arange(wl.B * per, dtype=np.int32).reshape(wl.B, per)], axis=1)
    return np.concatenate([kc, new]), np.concatenate([vc, new]), bt


def _first_child_target(T, V):
    """Target rows whose argmax at every node is the token of its first child,
    so the accepted path follows first children down to a leaf."""
    B, N = T["parent"].shape
    target = np.zeros((B, N, V), np.float32)
    for b in range(B):
        n = int(T["n"][b])
        for u in range(n):
            kids = [c for c in range(n) if int(T["parent"][b, c]) == u]
            target[b, u, int(T["token"][b, kids[0]]) if kids else 0] = 1.0
    return target


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_kv_commit_puts_each_accepted_node_at_its_position(layout):
    """After the commit, the row at context position pos[i] (stage 2's position
    of node i) holds node i's key and value for every node i of the accepted
    path, the context grows by acc_len + 1, and every other cache entry is
    unchanged."""
    wl, inp, T, _, f = _small_attention_case(3, layout)
    kc, vc, bt = _with_room(inp, wl, wl.K + 1)
    acc_len, acc_nodes, *_ = oracle.accept(_first_child_target(T, wl.V), T["n"], T["parent"], T["token"], wl.K)
    assert acc_len.max() >= 2   # a path deeper than the root is exercised
    kt, vt = f(inp.k_tree).astype(np.float64), f(inp.v_tree).astype(np.float64)
    k2, v2, ctx2 = oracle.kv_commit(kt, vt, acc_len, acc_nodes, kc, vc, inp.ctx_len, block_table=bt,
                                    page_size=wl.page_size)
    assert np.array_equal(ctx2, inp.ctx_len + acc_len + 1)
    touched_k = np.zeros(kc.shape[:-1], bool)
    for b in range(wl.B):
        for j in range(int(acc_len[b]) + 1):
            i = int(acc_nodes[b, j])
            p = int(T["pos"][b, i])
            assert T["depth"][b, i] == j and p == inp.ctx_len[b] + j
            for h in range(wl.Hkv):
                idx = (b, h, p) if bt is None else (int(bt[b, p // wl.page_size]), h, p % wl.page_size)
                assert np.array_equal(k2[idx], kt[b, i, h]) and np.array_equal(v2[idx], vt[b, i, h])
                touched_k[idx] = True
    assert np.array_equal(k2[~touched_k], kc[~touched_k]) and np.array_equal(v2[~touched_k], vc[~touched_k])


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_kv_commit_context_attention_equals_tree_attention(layout):
    """For every accepted node at depth j, plain attention of its query over the
    first ctx_len + j + 1 positions of the committed cache (keys gathered here
    by explicit page lookups, softmax by torch) equals the tree attention the
    verification pass computed for it: the committed prefix is exactly the key
    set that node saw."""
    wl, inp, T, out, f = _small_attention_case(5, layout)
    kc, vc, bt = _with_room(inp, wl, wl.K + 1)
    acc_len, acc_nodes, *_ = oracle.accept(_first_child_target(T, wl.V), T["n"], T["parent"], T["token"], wl.K)
    kt, vt, q = (f(a).astype(np.float64) for a in (inp.k_tree, inp.v_tree, inp.q))
    k2, v2, _ = oracle.kv_commit(kt, vt, acc_len, acc_nodes, kc, vc, inp.ctx_len, block_table=bt,
                                 page_size=wl.page_size)
    g = wl.Hq // wl.Hkv
    for b in range(wl.B):
        for j in range(int(acc_len[b]) + 1):
            i = int(acc_nodes[b, j])
            L = int(inp.ctx_len[b]) + j + 1
            for h in range(wl.Hq):
                kvh = h // g
                if bt is None:
                    ck, cv = k2[b, kvh, :L], v2[b, kvh, :L]
                else:
                    ck = np.stack([k2[bt[b, t // wl.page_size], kvh, t % wl.page_size] for t in range(L)])
                    cv = np.stack([v2[bt[b, t // wl.page_size], kvh, t % wl.page_size] for t in range(L)])
                np.testing.assert_allclose(_sdpa(q[b, i, h], ck, cv, inp.scale), out[b, i, h], rtol=1e-10,
                                           atol=1e-12)


# ---------------------------------------------------------------- drafter mask


def test_block_mask_bits_by_definition():
    """Bits written out from the definition (same block, inside n) for ragged
    n, a block that does not divide n, and rows past n."""
    n = np.array([1, 37, 70])
    m = oracle.block_mask(n, 80, 16)
    assert m.shape == (3, 80, 2) and m.dtype == np.uint64
    for b, nb in enumerate(n):
        for i in range(80):
            bits = {j for j in range(80) if (int(m[b, i, j // 64]) >> (j % 64)) & 1}
            want = {j for j in range(nb) if j // 16 == i // 16} if i < nb else set()
            assert bits == want, (b, i)


def test_masked_attention_with_ancestor_mask_is_tree_attention():
    """With stage 2's ancestor-or-self mask, masked attention reproduces the
    tree attention of the same tree (which walks parents instead)."""
    for layout in ("contiguous", "paged"):
        wl, inp, T, out, f = _small_attention_case(2, layout)
        got = oracle.masked_attention(f(inp.q), f(inp.k_tree), f(inp.v_tree), f(inp.k_ctx), f(inp.v_ctx),
                                      inp.ctx_len, T["mask"], T["n"], wl.Hkv, inp.scale,
                                      block_table=inp.block_table, page_size=wl.page_size)
        np.testing.assert_allclose(got, out, rtol=1e-12, atol=1e-13, equal_nan=True)


def test_one_block_is_unmasked_attention_and_unit_blocks_see_themselves():
    """A block spanning all n rows: every row attends to the whole context and
    every block position (torch SDPA without a mask); blocks of one with no
    context: each row's output is its own value row."""
    rng = np.random.default_rng(8)
    B, N, Hq, Hkv, d, L = 1, 12, 4, 2, 8, 9
    q = rng.standard_normal((B, N, Hq, d))
    kt, vt = rng.standard_normal((B, N, Hkv, d)), rng.standard_normal((B, N, Hkv, d))
    kc, vc = rng.standard_normal((B, Hkv, L, d)), rng.standard_normal((B, Hkv, L, d))
    n = np.array([10])
    out = oracle.masked_attention(q, kt, vt, kc, vc, np.array([L]), oracle.block_mask(n, N, 16), n, Hkv, 0.4)
    for i in range(10):
        for h in range(Hq):
            keys = np.concatenate([kc[0, h // 2], kt[0, :10, h // 2]])
            vals = np.concatenate([vc[0, h // 2], vt[0, :10, h // 2]])
            np.testing.assert_allclose(out[0, i, h], _sdpa(q[0, i, h], keys, vals, 0.4), rtol=1e-12, atol=1e-13)
    solo = oracle.masked_attention(q, kt, vt, kc, vc, np.array([0]), oracle.block_mask(n, N, 1), n, Hkv, 0.4)
    for i in range(10):
        for h in range(Hq):
            np.testing.assert_allclose(solo[0, i, h], vt[0, i, h // 2], rtol=1e-14)
    assert np.all(np.isnan(solo[0, 10:]))


# ---------------------------------------------------------------- confidence threshold


@pytest.mark.parametrize("seed", range(4))
def test_confidence_threshold_keeps_the_nodes_above_tau(seed):
    """Without a controller the threshold tree is the prefix of the fixed-budget
    tree made of its first n_min nodes and every further node with rho >= tau:
    best-first pops come in non-increasing rho (a child never beats its
    parent), so the nodes above tau are a prefix."""
    rng = np.random.default_rng(seed)
    K, k, V, n_max, n_min = 5, 4, 40, 60, 4
    x = rng.standard_normal((1, K, V)) * 2
    full, *_ = _tree_from_logits(x, k, n_max)
    rho = full[0].rho[:full[0].n]
    assert np.all(np.diff(rho) <= 1e-12 * rho[:-1])
    tried = 0
    for m in range(n_min + 1, len(rho) - 1, 7):
        if not rho[m - 1] > rho[m] * 1.001:
            continue
        tau = math.sqrt(rho[m - 1] * rho[m])   # strictly between node m-1 and node m
        t, *_ = _tree_from_logits(x, k, n_max, n_min=n_min, tau=tau)
        assert t[0].n == m == max(n_min, int((rho >= tau).sum()))
        for f in ("parent", "token", "depth"):
            assert np.array_equal(getattr(t[0], f)[:m], getattr(full[0], f)[:m]), f
        tried += 1
    assert tried >= 3
    # a threshold above every node leaves n_min nodes; tau = 0 is no threshold
    t, *_ = _tree_from_logits(x, k, n_max, n_min=n_min, tau=0.999)
    assert t[0].n == n_min
    t, *_ = _tree_from_logits(x, k, n_max, n_min=n_min, tau=0.0)
    assert t[0].n == n_max


def test_confidence_threshold_with_controller_stops_at_the_first_rule():
    """With the S(N) controller as well, the tree stops where the first of the
    two rules says so: n = min(n under S alone, n under tau alone)."""
    rng = np.random.default_rng(12)
    K, k, V, n_max, n_min = 6, 4, 30, 80, 3
    x = rng.standard_normal((2, K, V)) * 3
    n_grid = np.arange(n_max + 1, dtype=np.float64)
    C = (6.0 + 0.04 * n_grid + 0.15 * np.maximum(0, n_grid - 20)).astype(np.float32)
    s_only, *_ = _tree_from_logits(x, k, n_max, n_min=n_min, C=C)
    full, *_ = _tree_from_logits(x, k, n_max)
    tried = 0
    for b in range(2):
        rho = full[b].rho[:full[b].n]
        for m in (n_min + 2, s_only[b].n - 2, s_only[b].n + 5):
            if not (n_min < m < len(rho) and rho[m - 1] > rho[m] * 1.001):
                continue
            tau = math.sqrt(rho[m - 1] * rho[m])
            both, *_ = _tree_from_logits(x[b:b + 1], k, n_max, n_min=n_min, C=C, tau=tau)
            assert both[0].n == min(s_only[b].n, m), (b, m)
            tried += 1
    assert tried >= 3


# ---------------------------------------------------------------- latency calibration


def test_fit_recovers_a_noise_free_piecewise_model():
    N = np.array([1, 2, 4, 8, 16, 24, 32, 48, 64, 80, 96, 128, 160, 192, 224, 256])
    for (a, b, c, knee) in ((5.0, 0.03, 0.12, 64), (2.5, 0.0, 0.4, 20), (7.0, 0.05, 0.0, 300)):
        t = a + b * N + c * np.maximum(0, N - knee)
        fa, fb, fc, fk, sse = oracle.fit_verify_latency(N, t, 8, 200)
        assert sse < 1e-18
        pred = fa + fb * N + fc * np.maximum(0, N - fk)
        np.testing.assert_allclose(pred, t, rtol=1e-10, atol=1e-12)
        if c > 0:
            assert fk == knee and abs(fc - c) < 1e-9 and abs(fb - b) < 1e-9 and abs(fa - a) < 1e-9
        else:
            # no hinge in the data: every knee fits exactly, the smallest is kept
            assert abs(fc) < 1e-9 and fk == 8


def test_fit_is_the_least_squares_optimum():
    """Noisy data: at the chosen knee no (a, b, c) fits better (the gradient of
    the squared error vanishes there), and every other knee's own best fit
    (solved here from the normal equations) is no better."""
    rng = np.random.default_rng(3)
    N = np.arange(1, 257, 5)
    t = 4.0 + 0.02 * N + 0.3 * np.maximum(0, N - 97) + rng.normal(0, 0.2, N.size)
    a, b, c, knee, sse = oracle.fit_verify_latency(N, t, 10, 240)
    X = np.stack([np.ones(N.size), N, np.maximum(0, N - knee)], axis=1).astype(np.float64)
    r = t - X @ np.array([a, b, c])
    np.testing.assert_allclose(X.T @ r, 0.0, atol=1e-6)
    assert abs(sse - r @ r) < 1e-9 * max(1.0, sse)
    for k in range(10, 241):
        h = np.maximum(0, N - k).astype(np.float64)
        Xk = np.stack([np.ones(N.size), N.astype(np.float64)] + ([h] if h.any() else []), axis=1)
        coef = np.linalg.solve(Xk.T @ Xk, Xk.T @ t)
        rk = t - Xk @ coef
        assert rk @ rk >= sse * (1 - 1e-9)
    assert 90 <= knee <= 105


def test_latency_table_closed_form():
    C, L_AR = oracle.latency_table(3.0, 0.25, 0.5, 10, 1.5, 20)
    assert C.dtype == np.float32 and C.shape == (21,)
    assert C[0] == np.float32(4.5) and L_AR == np.float32(3.25)
    d = np.diff(C.astype(np.float64))
    np.testing.assert_allclose(d[:10], 0.25, rtol=1e-6)    # n = 1..10: slope b
    np.testing.assert_allclose(d[10:], 0.75, rtol=1e-6)    # past the knee: b + c
