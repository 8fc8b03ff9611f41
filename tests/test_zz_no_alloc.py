"""bastion_accept_noalloc: acceptance for callers that cannot allocate.

Some callers have no device allocator reachable when the step runs (their
memory is planned once at start-up), so they cannot provide the workspace
that bastion_accept takes.  bastion_accept_noalloc keeps that scratch in a
fixed array inside the library.  This file checks, through the C ABI, that it
returns exactly what bastion_accept returns, on two calls in a row (the
shared scratch must not carry state from one call into the next), that both
agree with the CPU oracle, and that sizes beyond its fixed array are refused.
It is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


def _outputs(B, N, K):
    return {k: torch.full(s, -7, dtype=torch.int32, device="cuda")
            for k, s in (("acc_len", (B,)), ("acc_nodes", (B, K + 1)), ("acc_tok", (B, K + 1)), ("bonus", (B,)),
                         ("argmax", (B, N)))}


def _case(name, seed, V):
    wl = I.WORKLOADS["controller_sweep_peaked"].scaled(name=name, B=4, V=V, n_min=1, n_max=48, L=64)
    inp, o = C.pick(wl, seed, with_attention=False)
    tree = o["tree"]
    target_h = C.target_for(inp, tree)
    want = C.oracle_accept(inp, tree, target_h)
    return wl, tree, C.dev(target_h, wl.dtype), want


# V = 30011: a bf16 row is not a multiple of 16 bytes, so the kernel reads it
# with plain loads; V = 30016: 16-byte rows, staged with bulk copies (the form
# the Qwen3- and Llama-sized vocabularies take)
CASES = (("noalloc_scalar", 0, 30011), ("noalloc_bulk", 1, 30016))


def test_noalloc_accept_matches_workspace_accept_twice_in_a_row():
    cases = [_case(*c) for c in CASES]
    for rep in range(2):
        for wl, tree, target, want in cases:
            B, N, K = wl.B, wl.n_max, wl.K
            n, par, tok = C.dev(tree["n"]), C.dev(tree["parent"]), C.dev(tree["token"])
            ref = _outputs(B, N, K)
            ws = torch.zeros(bn.bastion_accept_workspace_size(B, N), dtype=torch.uint8, device="cuda")
            bn.bastion_accept(target, n, par, tok, K, ref["acc_len"], ref["acc_nodes"], ref["acc_tok"], ref["bonus"],
                              ws, argmax_out=ref["argmax"])
            got = _outputs(B, N, K)
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            bn.bastion_accept_noalloc(target, n, par, tok, K, got["acc_len"], got["acc_nodes"], got["acc_tok"],
                                      got["bonus"], argmax_out=got["argmax"], dev_err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            for k in ref:   # integer outputs: exact, against the workspace call and against the oracle
                assert torch.equal(got[k], ref[k]), (rep, wl.name, k)
            for k, wv in zip(("acc_len", "acc_nodes", "acc_tok", "bonus", "argmax"), want):
                assert np.array_equal(got[k].cpu().numpy(), wv), (rep, wl.name, k)


def test_noalloc_accept_refuses_sizes_beyond_its_array():
    L = bn.lib()
    B, N = 128, 256          # 32768 argmax slots: more than the fixed array holds
    assert L.bastion_accept_workspace_size(B, N) > 128 * 1024
    P = ctypes.c_void_p(16)
    st = L.bastion_accept_noalloc(P, 1, B, N, 1000, 1000, 16, P, P, P, P, P, P, P, None, None, None)
    assert st == 2   # BASTION_ERR_UNSUPPORTED
    assert b"bastion_accept" in L.bastion_last_error()
