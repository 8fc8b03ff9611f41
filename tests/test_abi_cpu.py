"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function declared in include/bastion.h,
and reject bad arguments synchronously with the documented status, without
launching anything.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bastion.h")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, NO_DEVICE, DEVICE, TIMEOUT = 0, 1, 2, 3, 4, 5, 6, 7


@pytest.fixture(scope="module")
def L():
    from tree_speculative_decoding_bastion_gb300 import binding, build
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bastion_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_stages():
    names = declared_functions()
    for n in ("bastion_topk_softmax", "bastion_tree_build", "bastion_tree_attn", "bastion_accept"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_version_and_status_strings(L):
    assert L.bastion_abi_version() == 102
    for s, name in ((OK, b"BASTION_OK"), (INVALID, b"BASTION_ERR_INVALID_ARG"), (WORKSPACE, b"BASTION_ERR_WORKSPACE"),
                    (DEVICE, b"BASTION_ERR_DEVICE"), (TIMEOUT, b"BASTION_ERR_TIMEOUT")):
        assert L.bastion_status_string(s) == name
        assert L.bastion_status_str(s) == name


def test_error_word_helpers(L):
    from tree_speculative_decoding_bastion_gb300 import binding as bn
    assert L.bastion_error_status(0) == OK
    for bit in (bn.DEVERR_TOKEN, bn.DEVERR_N, bn.DEVERR_CTX, bn.DEVERR_PAGE, bn.DEVERR_LAYOUT):
        assert L.bastion_error_status(bit) == DEVICE
    assert L.bastion_error_status(bn.DEVERR_TIMEOUT) == TIMEOUT
    assert L.bastion_error_status(bn.DEVERR_TIMEOUT | bn.DEVERR_N) == TIMEOUT
    # NULL pointers are refused before any copy is enqueued
    assert L.bastion_read_error(None, ctypes.c_void_p(16), None) == INVALID
    assert L.bastion_read_error(ctypes.c_void_p(16), None, None) == INVALID
    assert L.bastion_topk_softmax_workspace_size(64, 151936, 8) == 0


P = ctypes.c_void_p(16)   # a non-NULL dummy; never dereferenced on these paths


def test_topk_softmax_rejects_bad_arguments(L):
    f = L.bastion_topk_softmax
    assert f(None, 1, 4, 1024, 1024, 4, P, P, P, P, None, None) == INVALID
    assert f(P, 7, 4, 1024, 1024, 4, P, P, P, P, None, None) == INVALID        # dtype
    assert f(P, 1, 4, 1024, 1000, 4, P, P, P, P, None, None) == INVALID        # row_stride < V
    assert f(P, 1, 0, 1024, 1024, 4, P, P, P, P, None, None) == INVALID        # rows
    assert f(P, 1, 4, 1024, 1024, 33, P, P, P, P, None, None) == UNSUPPORTED   # k > 32
    assert f(P, 1, 4, 3, 3, 4, P, P, P, P, None, None) == UNSUPPORTED          # k > V
    assert f(P, 1, 4, 300000, 300000, 4, P, P, P, P, None, None) == UNSUPPORTED  # V too large
    assert b"topk_softmax" in L.bastion_last_error()


def _tree_args(**kw):
    a = dict(ids=P, lg=P, lse=P, B=2, K=16, k=8, V=1000, root=P, ctx=P, n_min=8, n_max=64, C=None, L_AR=1.0)
    a.update(kw)
    return [a["ids"], a["lg"], a["lse"], a["B"], a["K"], a["k"], a["V"], a["root"], a["ctx"], a["n_min"],
            a["n_max"], a["C"], a["L_AR"]] + [P] * 9 + [None, None, None]


def test_tree_build_rejects_bad_arguments(L):
    f = L.bastion_tree_build
    assert f(*_tree_args(ids=None)) == INVALID
    assert f(*_tree_args(n_min=0)) == INVALID
    assert f(*_tree_args(n_min=65)) == INVALID
    assert f(*_tree_args(L_AR=0.0)) == INVALID
    assert f(*_tree_args(L_AR=float("nan"))) == INVALID
    assert f(*_tree_args(n_max=257, n_min=8)) == UNSUPPORTED
    assert f(*_tree_args(K=33)) == UNSUPPORTED
    assert f(*_tree_args(k=33)) == UNSUPPORTED


def test_tree_attn_rejects_bad_arguments(L):
    from tree_speculative_decoding_bastion_gb300.binding import KVCache
    kv = KVCache()
    kv.k = kv.v = 16
    kv.L_max = 4096
    f = L.bastion_tree_attn

    def call(**kw):
        a = dict(q=P, kt=P, vt=P, dt=1, B=1, N=64, Hq=32, Hkv=8, d=128, scale=0.088, kv=ctypes.byref(kv))
        a.update(kw)
        return f(a["q"], a["kt"], a["vt"], a["dt"], a["B"], a["N"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["kv"],
                 P, P, P, P, None, 0, None, None)

    assert call(q=None) == INVALID
    assert call(kv=None) == INVALID
    assert call(Hq=30) == INVALID            # Hq % Hkv
    assert call(scale=0.0) == INVALID
    assert call(d=96) == UNSUPPORTED
    assert call(N=300) == UNSUPPORTED
    kv.L_max = 0
    assert call() == INVALID
    kv.L_max = 4096
    kv.block_table = 16
    kv.max_pages, kv.num_pages, kv.page_size = 8, 8, 12
    assert call() == UNSUPPORTED              # page size must divide 128


def test_accept_rejects_bad_arguments(L):
    f = L.bastion_accept

    def call(**kw):
        a = dict(t=P, dt=1, B=2, N=64, V=1000, rs=1000, K=16, ws=P, wsb=1 << 20)
        a.update(kw)
        return f(a["t"], a["dt"], a["B"], a["N"], a["V"], a["rs"], a["K"], P, P, P, P, P, P, P, None, a["ws"],
                 a["wsb"], None, None)

    assert call(t=None) == INVALID
    assert call(rs=999) == INVALID
    assert call(ws=None) == INVALID
    assert call(V=300000, rs=300000) == UNSUPPORTED
    assert call(wsb=8) == WORKSPACE


def test_workspace_sizes_are_zero_without_a_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; sizes are device-dependent")
    assert L.bastion_accept_workspace_size(2, 64) >= 2 * 64 * 4
    assert L.bastion_init(0) == NO_DEVICE


def test_kv_commit_rejects_bad_arguments(L):
    from tree_speculative_decoding_bastion_gb300.binding import KVCache
    f = L.bastion_kv_commit
    kv = KVCache()
    kv.k, kv.v, kv.L_max = 16, 16, 4096

    def call(**kw):
        a = dict(kt=P, dt=1, B=2, N=64, H=8, d=128, K=16, ctx_out=P)
        a.update(kw)
        return f(a["kt"], P, a["dt"], a["B"], a["N"], a["H"], a["d"], a["K"], P, P, ctypes.byref(kv), P,
                 a["ctx_out"], None, None)

    assert call(kt=None) == INVALID
    assert call(ctx_out=None) == INVALID
    assert call(dt=5) == INVALID
    assert call(B=0) == INVALID
    assert call(N=300) == UNSUPPORTED
    assert call(K=33) == UNSUPPORTED
    assert call(d=4) == UNSUPPORTED            # 8 bytes per bf16 row: not a multiple of 16
    assert call(kt=ctypes.c_void_p(24)) == INVALID   # not 16-byte aligned
    kv.L_max = 0
    assert call() == INVALID
    kv.L_max = 4096
    kv.block_table = 16
    kv.max_pages, kv.num_pages, kv.page_size = 0, 8, 16
    assert call() == INVALID


def test_block_mask_rejects_bad_arguments(L):
    f = L.bastion_block_mask
    assert f(2, 64, 16, None, P, None, None) == INVALID
    assert f(2, 64, 16, P, None, None, None) == INVALID
    assert f(0, 64, 16, P, P, None, None) == INVALID
    assert f(2, 64, 0, P, P, None, None) == INVALID
    assert f(2, 300, 16, P, P, None, None) == UNSUPPORTED


def test_tree_build_threshold_rejects_bad_tau(L):
    f = L.bastion_tree_build_threshold

    def call(tau, ids=P):
        return f(ids, P, P, 2, 16, 8, 1000, P, P, 8, 64, None, ctypes.c_float(1.0), ctypes.c_float(tau), P, P, P, P,
                 P, P, P, P, P, None, None, None)

    assert call(0.5, ids=None) == INVALID
    assert call(-0.1) == INVALID
    assert call(1.5) == INVALID
    assert call(float("nan")) == INVALID
