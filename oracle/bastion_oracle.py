"""CPU oracle for the BASTION spec-tree step (test infrastructure only).

This module is the correctness reference for the CUDA library.  Only the test
suite, the smoke check and the benchmark's CPU-baseline leg may import it; the
product path never calls it and has no CPU fallback.  It imports numpy and
nothing from the CUDA package; the two share no code.

It is deliberately plain and slow: float64 arithmetic, straightforward loops,
library primitives (exp, stable sort, argmax, dot products) as single steps and
no blocking, fusion or reordering beyond what the definitions state.

Sources (cited by page title and section):
  [B] "Bastion: Budget-Aware Speculative Decoding with Tree-structured Block
      Diffusion Drafting", explainer page gist.science/de/paper/2605.29727
      (German) and its Spanish twin gist.science/es/paper/2605.29727.
      Section "Methodik: BASTION":
        §1 "Baumgestützte block-diffusionsbasierte Drafting": one drafter pass
           gives per-position marginals q_k(.); candidates at different
           positions combine freely into a prefix tree ("Randverteilungs-
           Unabhängigkeit"); path score rho(i) = prod_{k=1}^{d(i)} q_k(x_ik).
        §2 "Akzeptanz-Surrogat und Best-First-Erweiterung": A_hat(T) = sum of
           rho over the tree; best-first adds the valid node of highest rho.
        §3 "Hardwarebewusster Online-Budget-Controller": grow the tree until
           S(N) = A_hat(T_N) * L_AR / C(N) starts to fall.
      Section "Experimentelle Ergebnisse": greedy decoding (temperature 0).
      Section "Problemstellung": the target verifies the drafted tokens in one
      parallel pass ("baumgestützte Verifizierung" under "Akzeptanzlänge").

Readings where the pages are silent (each is listed in the design notes):
  * the root is node 0 of the tree and counts in N and in A_hat, rho(root) = 1
    (the empty product of §1);
  * children of a depth-d node are the top-k tokens of position d+1;
  * order: higher rho first, then lower token id, then lower parent index;
    rho is compared through its log, key = (fp32 sum of the path's logits,
    accumulated root to leaf) - (sum of the per-position log-normalisers),
    so exact ties at equal depth stay exact and the decision is taken in the
    kernel's precision; the reported rho uses the exact float64 path sum;
  * C(N) is a table indexed by N = 1..n_max; fixed budget when it is absent;
  * the controller pops unconditionally up to n_min, then stops at the first
    n with S(n+1) < S(n) (strict);
  * tree attention: node i attends to every context key and to the tree keys
    of its root-to-i path, self included, softmax(q.k * scale);
  * acceptance: per-node argmax (lowest id on ties), walk from the root to the
    child whose token equals the parent's argmax; accepted length counts the
    accepted draft tokens, the bonus is the argmax where the walk stops.

Every function here is pinned by CPU tests against closed forms, brute force,
library routines or worked examples; none is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------
# Stage 1: per-position marginals and top-k   ([B] Methodik §1)
# --------------------------------------------------------------------------


def marginals(logits_row: np.ndarray):
    """Softmax of one drafter position over the whole vocabulary, temperature 1.

    q(v) = exp(l_v - m) / sum_u exp(l_u - m), m = max_u l_u;  also returns
    lse = m + log sum_u exp(l_u - m) = log sum_u exp(l_u).
    [B] Methodik §1: the drafter yields per-position marginals q_k(.).
    """
    l = np.asarray(logits_row, dtype=np.float64)
    m = l.max()
    e = np.exp(l - m)
    z = e.sum()
    return e / z, m + math.log(z)


def topk_softmax(logits: np.ndarray, k: int):
    """Top-k candidates of every drafter row.

    ``logits`` is [R, V] (any float dtype; values are taken exactly).  Returns
    ids [R,k] int32, lg [R,k] float64 (the logits), q [R,k] float64 and
    lse [R] float64.  Candidates are ordered by logit descending, then token id
    ascending (a stable sort of -logit), which is the order of q as well.
    """
    L = np.asarray(logits, dtype=np.float64)
    R, V = L.shape
    ids = np.empty((R, k), dtype=np.int32)
    lg = np.empty((R, k), dtype=np.float64)
    q = np.empty((R, k), dtype=np.float64)
    lse = np.empty(R, dtype=np.float64)
    for r in range(R):
        q_full, lse[r] = marginals(L[r])
        order = np.argsort(-L[r], kind="stable")[:k]
        ids[r] = order
        lg[r] = L[r, order]
        q[r] = q_full[order]
    return ids, lg, q, lse


# --------------------------------------------------------------------------
# Stage 2: best-first prefix tree with the S(N) budget stop
#          ([B] Methodik §1 "Pfad-Bewertung", §2, §3)
# --------------------------------------------------------------------------


@dataclass
class Tree:
    n: int
    parent: np.ndarray      # [n_max] int32, -1 for the root and unused rows
    token: np.ndarray       # [n_max] int32
    depth: np.ndarray       # [n_max] int32
    pos: np.ndarray         # [n_max] int32  (ctx_len + depth)
    rho: np.ndarray         # [n_max] float64
    mask: np.ndarray        # [n_max, W] uint64 ancestor-or-self bits
    ahat: float             # A_hat(T_n)
    S: float                # S(n)
    S_curve: np.ndarray     # [n_max] float64, S(j+1) for j < n, 0 beyond
    key: np.ndarray         # [n_max] float64 log rho of each node (diagnostic)
    min_gap: float          # smallest relative gap of an inexact decision


def _build_one(ids, lg, lse, root_tok, ctx_len, n_min, n_max, C, L_AR, tau=0.0) -> Tree:
    K, k = ids.shape
    # prefix of log-normalisers: P[d] = sum_{t=1..d} lse_t, so that
    # log rho(i) = sum_{t<=d} l_t(x_t) - P[d]   (log of the product in §1)
    P = np.zeros(K + 1, dtype=np.float64)
    for t in range(1, K + 1):
        P[t] = P[t - 1] + float(lse[t - 1])

    par = [-1]
    tok = [int(root_tok)]
    dep = [0]
    S32 = [np.float32(0.0)]          # fp32 logit sum along the path (decisions)
    S64 = [0.0]                      # exact float64 logit sum along the path (reported rho)
    key = [0.0]                      # log rho(root) = log 1
    rho = [1.0]

    # frontier: every child of every tree node not yet in the tree
    f_key: list = []
    f_tok: list = []
    f_par: list = []
    f_dep: list = []
    f_S: list = []
    f_S64: list = []

    def offer_children(i: int) -> None:
        d = dep[i]
        if d >= K:
            return
        for j in range(k):
            s = np.float32(S32[i] + np.float32(lg[d, j]))    # position d+1
            f_key.append(float(s) - P[d + 1])
            f_tok.append(int(ids[d, j]))
            f_par.append(i)
            f_dep.append(d + 1)
            f_S.append(s)
            f_S64.append(S64[i] + float(lg[d, j]))

    offer_children(0)
    ahat = [1.0]                     # A_hat after n nodes, n = 1 (root only)
    min_gap = math.inf

    def best_index() -> int:
        # highest rho (key), then lowest token id, then lowest parent index
        order = np.lexsort((np.asarray(f_par), np.asarray(f_tok), -np.asarray(f_key)))
        return int(order[0])

    def decision_gap(b: int) -> float:
        # relative rho gap between the chosen candidate and every other one
        # whose order is not an exact tie (same depth, same fp32 logit sum)
        fk = np.asarray(f_key)
        exact_tie = (np.asarray(f_dep) == f_dep[b]) & (np.asarray(f_S, dtype=np.float32) == f_S[b])
        others = fk[~exact_tie]
        if others.size == 0:
            return math.inf
        return 1.0 - math.exp(min(0.0, float(others.max()) - f_key[b]))

    while len(par) < n_max and f_key:
        n = len(par)
        b = best_index()
        min_gap = min(min_gap, decision_gap(b))
        rho_next = math.exp(f_S64[b] - P[f_dep[b]])
        if tau > 0.0 and n >= n_min:
            # cumulative draft confidence below the threshold: stop (FlexDraft
            # page, "Flex-Decoding", selective verification).  Decided on the
            # fp32 log rho (fp32 logit sum minus the float64 lse prefix, rounded
            # to fp32) against log tau rounded to fp32.
            min_gap = min(min_gap, 1.0 - math.exp(-abs(f_key[b] - math.log(tau))))
            if np.float32(float(f_S[b]) - P[f_dep[b]]) < np.float32(math.log(tau)):
                break
        if C is not None and n >= n_min:
            s_now = ahat[-1] * L_AR / float(C[n])
            s_next = (ahat[-1] + rho_next) * L_AR / float(C[n + 1])
            min_gap = min(min_gap, abs(s_next - s_now) / max(s_now, s_next))
            if s_next < s_now:       # S(N) begins to fall: stop (§3)
                break
        # pop candidate b into the tree
        par.append(f_par[b])
        tok.append(f_tok[b])
        dep.append(f_dep[b])
        S32.append(f_S[b])
        S64.append(f_S64[b])
        key.append(f_key[b])
        rho.append(rho_next)
        ahat.append(ahat[-1] + rho_next)
        for lst in (f_key, f_tok, f_par, f_dep, f_S, f_S64):
            del lst[b]
        offer_children(len(par) - 1)

    n = len(par)
    W = (n_max + 63) // 64
    out_par = np.full(n_max, -1, dtype=np.int32)
    out_tok = np.full(n_max, -1, dtype=np.int32)
    out_dep = np.full(n_max, -1, dtype=np.int32)
    out_pos = np.full(n_max, -1, dtype=np.int32)
    out_rho = np.zeros(n_max, dtype=np.float64)
    out_key = np.zeros(n_max, dtype=np.float64)
    mask = np.zeros((n_max, W), dtype=np.uint64)
    S_curve = np.zeros(n_max, dtype=np.float64)
    for i in range(n):
        out_par[i], out_tok[i], out_dep[i] = par[i], tok[i], dep[i]
        out_pos[i] = int(ctx_len) + dep[i]
        out_rho[i] = rho[i]
        out_key[i] = key[i]
        j = i
        while j >= 0:                # ancestor-or-self bits
            mask[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
            j = par[j]
        c = 1.0 if C is None else float(C[i + 1])
        S_curve[i] = ahat[i] * L_AR / c
    return Tree(n=n, parent=out_par, token=out_tok, depth=out_dep, pos=out_pos, rho=out_rho,
                mask=mask, ahat=ahat[n - 1], S=S_curve[n - 1], S_curve=S_curve, key=out_key,
                min_gap=min_gap)


def tree_build(ids, lg, lse, root_tok, ctx_len, n_min: int, n_max: int,
               C: Optional[np.ndarray], L_AR: float, tau: float = 0.0) -> list:
    """Best-first tree of every request.

    ids/lg are [B, K, k] (top-k of each position, in stage-1 order), lse is
    [B, K].  ``C`` is the latency table C[0..n_max] (entry n is C(n)) or None for
    a fixed budget (then S(n) is reported with C = 1).  ``tau`` > 0 adds the
    confidence threshold of the FlexDraft page ("Flex-Decoding", selective
    verification): past n_min the tree also stops at the first node whose
    rho (the cumulative draft confidence of its path) is below tau.  Returns
    one Tree per request.
    """
    ids = np.asarray(ids)
    lg = np.asarray(lg, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    return [_build_one(ids[b], lg[b], lse[b], root_tok[b], ctx_len[b], n_min, n_max, C, L_AR, tau)
            for b in range(ids.shape[0])]


def stack_trees(trees: Sequence[Tree]) -> dict:
    """Batch the per-request trees into [B, ...] arrays."""
    return {
        "n": np.array([t.n for t in trees], dtype=np.int32),
        "parent": np.stack([t.parent for t in trees]),
        "token": np.stack([t.token for t in trees]),
        "depth": np.stack([t.depth for t in trees]),
        "pos": np.stack([t.pos for t in trees]),
        "rho": np.stack([t.rho for t in trees]),
        "mask": np.stack([t.mask for t in trees]),
        "ahat": np.array([t.ahat for t in trees]),
        "S": np.array([t.S for t in trees]),
        "S_curve": np.stack([t.S_curve for t in trees]),
        "min_gap": min(t.min_gap for t in trees),
        "gaps": np.array([t.min_gap for t in trees]),
    }


# --------------------------------------------------------------------------
# Stage 3: tree-masked verification attention   ([B] Problemstellung,
#          "baumgestützte Verifizierung")
# --------------------------------------------------------------------------


def path_to_root(parent: np.ndarray, i: int) -> list:
    """Node indices root -> i (depth order)."""
    p = []
    while i >= 0:
        p.append(i)
        i = int(parent[i])
    return p[::-1]


def context_kv(k_ctx, v_ctx, block_table, b: int, kvh: int, L: int, page_size: int):
    """The first L context keys/values of request b, KV head kvh, as float64."""
    if block_table is None:
        return (np.asarray(k_ctx[b, kvh, :L], dtype=np.float64),
                np.asarray(v_ctx[b, kvh, :L], dtype=np.float64))
    pages = [int(block_table[b, t // page_size]) for t in range(0, L, page_size)]
    kk = np.concatenate([np.asarray(k_ctx[p, kvh], dtype=np.float64) for p in pages])[:L]
    vv = np.concatenate([np.asarray(v_ctx[p, kvh], dtype=np.float64) for p in pages])[:L]
    return kk, vv


def attend(qv: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """softmax(keys . q * scale) . values in float64 (one query row)."""
    s = keys @ np.asarray(qv, dtype=np.float64) * scale
    m = s.max()
    p = np.exp(s - m)
    return (p @ values) / p.sum()


def tree_attention(q, k_tree, v_tree, k_ctx, v_ctx, ctx_len, parent, n, Hkv: int, scale: float,
                   block_table=None, page_size: int = 16, rows=None) -> np.ndarray:
    """Attention of every tree node over context ∪ its root path.

    q [B, n_max, Hq, d]; k_tree/v_tree [B, n_max, Hkv, d]; k_ctx/v_ctx as
    contiguous [B, Hkv, L, d] or paged [P, Hkv, page, d] with block_table.
    For node i < n[b] and query head h (KV head h // (Hq/Hkv)) the key list is
    context positions 0..ctx_len[b]-1 followed by the tree nodes on the path
    root -> i.  Returns [B, n_max, Hq, d] float64 with NaN for rows not computed.
    ``rows`` optionally restricts the work to a list of (b, i, h).
    """
    B, N, Hq, d = q.shape
    g = Hq // Hkv
    out = np.full((B, N, Hq, d), np.nan, dtype=np.float64)
    if rows is None:
        rows = [(b, i, h) for b in range(B) for i in range(int(n[b])) for h in range(Hq)]
    cache = {}
    # visit rows grouped by (request, KV head) so each context is read once
    for (b, i, h) in sorted(rows, key=lambda r: (r[0], r[2] // g, r[1], r[2])):
        kvh = h // g
        if (b, kvh) not in cache:
            cache.clear()
            cache[(b, kvh)] = context_kv(k_ctx, v_ctx, block_table, b, kvh, int(ctx_len[b]), page_size)
        kc, vc = cache[(b, kvh)]
        path = path_to_root(parent[b], i)
        kt = np.asarray(k_tree[b, path, kvh], dtype=np.float64)
        vt = np.asarray(v_tree[b, path, kvh], dtype=np.float64)
        keys = np.concatenate([kc, kt])
        values = np.concatenate([vc, vt])
        out[b, i, h] = attend(q[b, i, h], keys, values, scale)
    return out


# --------------------------------------------------------------------------
# Stage 4: greedy acceptance   ([B] Experimentelle Ergebnisse: temperature 0;
#          Akzeptanzlänge)
# --------------------------------------------------------------------------


def accept(target, n, parent, token, K: int):
    """Greedy verification of every request's tree.

    target [B, n_max, V] (values taken exactly).  a_i = argmax_v target[b,i,v]
    (lowest id on ties) for i < n[b].  Starting at the root, move to the child
    whose token equals a_u; stop when there is none, the bonus token is a_u.
    Returns acc_len [B], acc_nodes [B, K+1] (root first, -1 padded),
    acc_tok [B, K+1] (accepted draft tokens then the bonus, -1 padded),
    bonus [B] and argmax [B, n_max] (-1 for rows >= n[b]).
    """
    B, N, V = target.shape
    acc_len = np.zeros(B, dtype=np.int32)
    acc_nodes = np.full((B, K + 1), -1, dtype=np.int32)
    acc_tok = np.full((B, K + 1), -1, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    amax = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        nb = int(n[b])
        for i in range(nb):
            amax[b, i] = int(np.argmax(np.asarray(target[b, i], dtype=np.float64)))
        u = 0
        path = [0]
        toks = []
        while True:
            a = int(amax[b, u])
            nxt = -1
            for v in range(nb):
                if int(parent[b, v]) == u and int(token[b, v]) == a:
                    nxt = v
                    break
            if nxt < 0:
                break
            u = nxt
            path.append(u)
            toks.append(a)
        acc_len[b] = len(path) - 1
        acc_nodes[b, : len(path)] = path
        acc_tok[b, : len(toks)] = toks
        acc_tok[b, len(toks)] = int(amax[b, u])
        bonus[b] = int(amax[b, u])
    return acc_len, acc_nodes, acc_tok, bonus, amax


# --------------------------------------------------------------------------
# After acceptance: commit the accepted path's keys and values to the context
# cache   (FlexDraft page, "Flex-Decoding", decoupled execution: the next draft
#          reuses the KV cache of the verification pass; [B] "Das Ergebnis":
#          each step's accepted tokens extend the text)
# --------------------------------------------------------------------------


def kv_commit(k_tree, v_tree, acc_len, acc_nodes, k_ctx, v_ctx, ctx_len, block_table=None, page_size: int = 16):
    """The context cache after the accepted path of every request joins it.

    For request b with a = acc_len[b] and c = ctx_len[b], the path's nodes
    acc_nodes[b, 0..a] (root first: the root is the token the previous step
    emitted, followed by the a accepted draft tokens) are appended at context
    positions c .. c+a of every KV head, and the context grows to c + a + 1.
    The root's keys were computed in the verification pass (tree node 0), so
    it is committed with the accepted drafts; the bonus token becomes the
    next step's root.

    k_tree/v_tree [B, n_max, Hkv, d]; k_ctx/v_ctx contiguous [B, Hkv, L, d] or
    paged [P, Hkv, page_size, d] with block_table [B, max_pages] (position p of
    request b lives in page block_table[b, p // page_size], slot
    p % page_size).  Returns (k_ctx', v_ctx', ctx_len') as new arrays; the
    inputs are not modified.
    """
    k_new = np.array(k_ctx, copy=True)
    v_new = np.array(v_ctx, copy=True)
    B, _, Hkv, _ = np.shape(k_tree)
    ctx_new = np.array(ctx_len, dtype=np.int32, copy=True)
    for b in range(B):
        a = int(acc_len[b])
        c = int(ctx_len[b])
        for j in range(a + 1):
            node = int(acc_nodes[b, j])
            p = c + j
            for h in range(Hkv):
                if block_table is None:
                    k_new[b, h, p] = k_tree[b, node, h]
                    v_new[b, h, p] = v_tree[b, node, h]
                else:
                    page = int(block_table[b, p // page_size])
                    k_new[page, h, p % page_size] = k_tree[b, node, h]
                    v_new[page, h, p % page_size] = v_tree[b, node, h]
        ctx_new[b] = c + a + 1
    return k_new, v_new, ctx_new


# --------------------------------------------------------------------------
# Block-diffusion drafter mask   (FlexDraft page, "Attention-Tuning": mask
#          tokens appended to the clean prefix attend bidirectionally inside
#          their block and to the clean prefix, and stay isolated from other
#          blocks; BASTION Methodik §1: the drafter fills a block of positions
#          in one pass)
# --------------------------------------------------------------------------


def block_mask(n, n_max: int, block: int) -> np.ndarray:
    """uint64 [B, n_max, ceil(n_max/64)]: for request b and row i < n[b], bit j
    is set iff j < n[b] and j and i lie in the same block of `block`
    consecutive positions (i // block == j // block); rows i >= n[b] are 0."""
    B = len(n)
    W = (n_max + 63) // 64
    mask = np.zeros((B, n_max, W), dtype=np.uint64)
    for b in range(B):
        nb = int(n[b])
        for i in range(nb):
            for j in range(nb):
                if i // block == j // block:
                    mask[b, i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return mask


def masked_attention(q, k_tree, v_tree, k_ctx, v_ctx, ctx_len, mask, n, Hkv: int, scale: float,
                     block_table=None, page_size: int = 16, rows=None) -> np.ndarray:
    """Attention of rows i < n[b] over the context and the positions j whose
    bit is set in mask[b, i] (ascending j), float64; NaN for rows not computed.
    Shapes as in tree_attention; ``rows`` optionally lists the (b, i, h) to do."""
    B, N, Hq, d = q.shape
    g = Hq // Hkv
    out = np.full((B, N, Hq, d), np.nan, dtype=np.float64)
    if rows is None:
        rows = [(b, i, h) for b in range(B) for i in range(int(n[b])) for h in range(Hq)]
    cache = {}
    for (b, i, h) in sorted(rows, key=lambda r: (r[0], r[2] // g, r[1], r[2])):
        kvh = h // g
        if (b, kvh) not in cache:
            cache.clear()
            cache[(b, kvh)] = context_kv(k_ctx, v_ctx, block_table, b, kvh, int(ctx_len[b]), page_size)
        kc, vc = cache[(b, kvh)]
        sel = [j for j in range(N) if (int(mask[b, i, j // 64]) >> (j % 64)) & 1]
        keys = np.concatenate([kc, np.asarray(k_tree[b, sel, kvh], dtype=np.float64)])
        values = np.concatenate([vc, np.asarray(v_tree[b, sel, kvh], dtype=np.float64)])
        out[b, i, h] = attend(q[b, i, h], keys, values, scale)
    return out


# --------------------------------------------------------------------------
# Latency-table calibration   ([B] Methodik §3: the controller needs C(N), the
#          cost of a step that verifies N tree tokens, and L_AR; the pages
#          model the verification latency from memory bandwidth and compute,
#          calibrated on observed runtimes of the device)
# --------------------------------------------------------------------------

KNEE_TIE_RTOL = 1e-9


def fit_verify_latency(N, t, knee_lo: int, knee_hi: int):
    """Least-squares fit of t ≈ a + b N + c max(0, N - knee) for every integer
    knee in [knee_lo, knee_hi]; returns (a, b, c, knee, sse) of the knee with
    the smallest squared error (the smallest such knee when several lie within
    1e-9 of the minimum, relative, or 1e-12 of sum t^2).  A knee at or past every N leaves the
    hinge column zero: that fit is (a, b) alone with c = 0 (as is a knee whose
    hinge column is a combination of 1 and N).  Needs two distinct N."""
    N = np.asarray(N, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    if np.unique(N).size < 2:
        raise ValueError("the fit needs at least two distinct N")
    line = np.stack([np.ones_like(N), N], axis=1)
    fits = []
    for knee in range(knee_lo, knee_hi + 1):
        hinge = np.maximum(0.0, N - knee)
        # the hinge is used only where it is not (to 1e-9 of its norm) a
        # combination of 1 and N: every N on one side of the knee, or a single
        # N at the knee, makes the fit a straight line with c = 0
        use = False
        if np.any(hinge > 0):
            proj, *_ = np.linalg.lstsq(line, hinge, rcond=None)
            use = np.linalg.norm(hinge - line @ proj) > 1e-9 * np.linalg.norm(hinge)
        cols = [np.ones_like(N), N] + ([hinge] if use else [])
        A = np.stack(cols, axis=1)
        coef, *_ = np.linalg.lstsq(A, t, rcond=None)
        r = t - A @ coef
        a, b = float(coef[0]), float(coef[1])
        c = float(coef[2]) if len(cols) == 3 else 0.0
        fits.append((float(r @ r), knee, a, b, c))
    # ties: within 1e-9 of the minimum, relative, or 1e-12 of the data's
    # energy sum t^2 (fits that differ by rounding only, e.g. data without a
    # hinge, where every knee past the data fits exactly)
    best = min(f[0] for f in fits)
    tol = best * KNEE_TIE_RTOL + 1e-12 * float(t @ t)
    sse, knee, a, b, c = next(f for f in fits if f[0] <= best + tol)
    return a, b, c, knee, sse


def latency_table(a: float, b: float, c: float, knee: int, t_draft: float, n_max: int):
    """C[n] = t_draft + a + b n + c max(0, n - knee) for n = 0..n_max (float32,
    the stage-2 table) and L_AR = T_verify(1) = a + b + c max(0, 1 - knee), the
    cost of a plain autoregressive step (one token verified)."""
    n = np.arange(n_max + 1, dtype=np.float64)
    C = (t_draft + a + b * n + c * np.maximum(0.0, n - knee)).astype(np.float32)
    L_AR = float(np.float32(a + b + c * max(0.0, 1.0 - knee)))
    return C, L_AR
