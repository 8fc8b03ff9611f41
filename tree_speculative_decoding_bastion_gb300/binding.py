"""Python binding of the C ABI in ``include/bastion.h`` (argument marshalling only).

Every function here takes torch CUDA tensors, checks their dtype/shape/device,
and passes raw pointers, sizes and the current CUDA stream to
``libbastion.so``.  All computation happens in the library's kernels; there is
no CPU or PyTorch fallback.  If the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbastion.so")

BASTION_F32 = 0
BASTION_BF16 = 1
DEVERR_TOKEN = 0x1
DEVERR_N = 0x2
DEVERR_CTX = 0x4
DEVERR_PAGE = 0x8
DEVERR_TIMEOUT = 0x10
DEVERR_LAYOUT = 0x20

_c_int, _c_i64, _c_f, _c_p, _c_sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class BastionError(RuntimeError):
    pass


class KVCache(ctypes.Structure):
    """Mirror of ``bastion_kv_cache``."""
    _fields_ = [("k", _c_p), ("v", _c_p), ("L_max", _c_i64), ("block_table", _c_p),
                ("max_pages", _c_int), ("num_pages", _c_int), ("page_size", _c_int)]


_SIGS = {
    "bastion_abi_version": (_c_int, []),
    "bastion_status_string": (ctypes.c_char_p, [_c_int]),
    "bastion_status_str": (ctypes.c_char_p, [_c_int]),
    "bastion_read_error": (_c_int, [_c_p, _c_p, _c_p]),
    "bastion_error_status": (_c_int, [ctypes.c_uint32]),
    "bastion_topk_softmax_workspace_size": (_c_sz, [_c_int, _c_int, _c_int]),
    "bastion_last_error": (ctypes.c_char_p, []),
    "bastion_init": (_c_int, [_c_int]),
    "bastion_topk_softmax": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p,
                                      _c_p]),
    "bastion_tree_build": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_int, _c_int,
                                    _c_p, _c_f, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                    _c_p]),
    "bastion_tree_build_threshold": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_int,
                                              _c_int, _c_p, _c_f, _c_f, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                              _c_p, _c_p, _c_p, _c_p, _c_p]),
    "bastion_tree_attn_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(KVCache)]),
    "bastion_tree_attn": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f,
                                   ctypes.POINTER(KVCache), _c_p, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "bastion_accept_workspace_size": (_c_sz, [_c_int, _c_int]),
    "bastion_accept": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p,
                                _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "bastion_accept_noalloc": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_p, _c_p, _c_p,
                                        _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "bastion_kv_commit": (_c_int, [_c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p,
                                   ctypes.POINTER(KVCache), _c_p, _c_p, _c_p, _c_p]),
    "bastion_block_mask": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p]),
    "bastion_fit_verify_latency": (_c_int, [_c_p, _c_p, _c_int, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "bastion_latency_table": (_c_int, [_c_p, ctypes.c_int32, ctypes.c_double, _c_int, _c_p, _c_p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libbastion.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise BastionError(f"{LIB_PATH} is missing: build it with "
                               "`python -m tree_speculative_decoding_bastion_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        L = lib()
        raise BastionError(f"{what}: {L.bastion_status_string(status).decode()} "
                           f"({L.bastion_last_error().decode()})")


# While a step is being prepared (SpecTreeStep.prepare), the stage functions
# record their marshalled calls here instead of issuing them.
_rec = threading.local()


def _call(name: str, *args) -> None:
    """Issue library call `name` with its marshalled arguments, or record it
    when a step is being prepared on this thread."""
    fn = getattr(lib(), name)
    calls = getattr(_rec, "calls", None)
    if calls is not None:
        calls.append((fn, args, name))
        return
    _check(fn(*args), name)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return BASTION_F32
    if t.dtype == torch.bfloat16:
        return BASTION_BF16
    raise BastionError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _need(t: torch.Tensor, dtype, shape, name: str) -> None:
    if not t.is_cuda:
        raise BastionError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise BastionError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise BastionError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise BastionError(f"{name} must be contiguous")


def bastion_init(device: int = 0) -> None:
    _check(lib().bastion_init(int(device)), "bastion_init")


def bastion_read_error(dev_err: torch.Tensor, stream=None) -> int:
    """The device error word (int32/uint32 [1] on the device): the library
    enqueues the copy on `stream`, this helper then waits for that stream and
    returns the word (BASTION_DEVERR_* bits)."""
    _need(dev_err, None, (1,), "dev_err")
    host = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().bastion_read_error(_ptr(dev_err), ctypes.c_void_p(host.data_ptr()), ctypes.c_void_p(s.cuda_stream)),
           "bastion_read_error")
    s.synchronize()
    return int(host.item()) & 0xFFFFFFFF


def bastion_error_status(word: int) -> int:
    """Status of an error word: 0 OK, 6 bad data, 7 an in-kernel wait expired."""
    return int(lib().bastion_error_status(int(word) & 0xFFFFFFFF))


def bastion_topk_softmax(logits: torch.Tensor, k: int, ids, lg, q, lse, dev_err=None, stream=None) -> None:
    """Stage 1. logits [rows, V] (rows of a [B, K, V] tensor) f32/bf16 with unit
    element stride; ids int32 [rows, k], lg/q float32 [rows, k], lse float64 [rows]."""
    if logits.dim() < 2 or logits.stride(-1) != 1:
        raise BastionError("logits must be [..., V] with contiguous rows")
    V = logits.shape[-1]
    flat = logits.reshape(-1, V)
    rows = flat.shape[0]
    row_stride = flat.stride(0)
    for t, dt, name in ((ids, torch.int32, "ids"), (lg, torch.float32, "lg"), (q, torch.float32, "q")):
        _need(t, dt, None, name)
        if t.numel() != rows * k:
            raise BastionError(f"{name} must hold rows*k = {rows * k} elements")
    _need(lse, torch.float64, None, "lse")
    if lse.numel() != rows:
        raise BastionError("lse must hold one value per row")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    _call("bastion_topk_softmax", _ptr(flat), _dtype_code(logits), rows, V, row_stride, int(k), _ptr(ids), _ptr(lg),
          _ptr(q), _ptr(lse), _ptr(dev_err), _stream(stream))


def bastion_tree_build(ids, lg, lse, V: int, root_tok, ctx_len, n_min: int, n_max: int, C: Optional[torch.Tensor],
                       L_AR: float, n, parent, token, depth, pos, rho, mask, ahat, S, S_curve=None, dev_err=None,
                       stream=None, tau: float = 0.0) -> None:
    """Stage 2. ids int32 / lg float32 [B, K, k]; lse float64 [B, K]; root_tok, ctx_len int32 [B];
    C float32 [n_max+1] or None (fixed budget); tau > 0 adds the confidence
    threshold (bastion_tree_build_threshold). Outputs as in bastion.h."""
    B, K, k = ids.shape
    _need(ids, torch.int32, (B, K, k), "ids")
    _need(lg, torch.float32, (B, K, k), "lg")
    _need(lse, torch.float64, (B, K), "lse")
    _need(root_tok, torch.int32, (B,), "root_tok")
    _need(ctx_len, torch.int32, (B,), "ctx_len")
    if C is not None:
        _need(C, torch.float32, (n_max + 1,), "C")
    W = (n_max + 63) // 64
    _need(n, torch.int32, (B,), "n")
    for t, name in ((parent, "parent"), (token, "token"), (depth, "depth"), (pos, "pos")):
        _need(t, torch.int32, (B, n_max), name)
    _need(rho, torch.float32, (B, n_max), "rho")
    _need(mask, torch.int64, (B, n_max, W), "mask")
    _need(ahat, torch.float32, (B,), "ahat")
    _need(S, torch.float32, (B,), "S")
    if S_curve is not None:
        _need(S_curve, torch.float32, (B, n_max), "S_curve")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    if tau:
        _call("bastion_tree_build_threshold", _ptr(ids), _ptr(lg), _ptr(lse), B, K, k, int(V), _ptr(root_tok),
              _ptr(ctx_len), int(n_min), int(n_max), _ptr(C), float(L_AR), float(tau), _ptr(n), _ptr(parent),
              _ptr(token), _ptr(depth), _ptr(pos), _ptr(rho), _ptr(mask), _ptr(ahat), _ptr(S), _ptr(S_curve),
              _ptr(dev_err), _stream(stream))
        return
    _call("bastion_tree_build", _ptr(ids), _ptr(lg), _ptr(lse), B, K, k, int(V), _ptr(root_tok), _ptr(ctx_len),
          int(n_min), int(n_max), _ptr(C), float(L_AR), _ptr(n), _ptr(parent), _ptr(token), _ptr(depth), _ptr(pos),
          _ptr(rho), _ptr(mask), _ptr(ahat), _ptr(S), _ptr(S_curve), _ptr(dev_err), _stream(stream))


@dataclass
class KV:
    """Context KV cache: contiguous (k, v [B, Hkv, L_max, d]) or paged
    (k, v [num_pages, Hkv, page_size, d] + block_table int32 [B, max_pages])."""
    k: torch.Tensor
    v: torch.Tensor
    block_table: Optional[torch.Tensor] = None

    def c_struct(self) -> KVCache:
        s = KVCache()
        s.k = self.k.data_ptr()
        s.v = self.v.data_ptr()
        if self.block_table is None:
            s.L_max = self.k.shape[2]
            s.block_table = None
            s.max_pages = s.num_pages = s.page_size = 0
        else:
            s.L_max = 0
            s.block_table = self.block_table.data_ptr()
            s.max_pages = self.block_table.shape[1]
            s.num_pages = self.k.shape[0]
            s.page_size = self.k.shape[2]
        return s


def bastion_tree_attn_workspace_size(B: int, n_max: int, Hq: int, Hkv: int, d: int, kv: KV) -> int:
    s = kv.c_struct()
    return int(lib().bastion_tree_attn_workspace_size(B, n_max, Hq, Hkv, d, ctypes.byref(s)))


def bastion_tree_attn(q, k_tree, v_tree, kv: KV, ctx_len, mask, n, out, scale: float, ws=None, dev_err=None,
                      stream=None) -> None:
    """Stage 3. q/out [B, n_max, Hq, d]; k_tree/v_tree [B, n_max, Hkv, d] (same dtype, f32 or bf16)."""
    B, N, Hq, d = q.shape
    Hkv = k_tree.shape[2]
    dt = q.dtype
    _need(q, dt, None, "q")
    _need(out, dt, (B, N, Hq, d), "out")
    _need(k_tree, dt, (B, N, Hkv, d), "k_tree")
    _need(v_tree, dt, (B, N, Hkv, d), "v_tree")
    _need(kv.k, dt, None, "kv.k")
    _need(kv.v, dt, tuple(kv.k.shape), "kv.v")
    if kv.block_table is not None:
        _need(kv.block_table, torch.int32, None, "block_table")
    _need(ctx_len, torch.int32, (B,), "ctx_len")
    _need(n, torch.int32, (B,), "n")
    _need(mask, torch.int64, (B, N, (N + 63) // 64), "mask")
    if ws is not None:
        _need(ws, torch.uint8, None, "ws")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    s = kv.c_struct()
    _call("bastion_tree_attn", _ptr(q), _ptr(k_tree), _ptr(v_tree), _dtype_code(q), B, N, Hq, Hkv, d, float(scale),
          ctypes.pointer(s), _ptr(ctx_len), _ptr(mask), _ptr(n), _ptr(out), _ptr(ws),
          0 if ws is None else ws.numel(), _ptr(dev_err), _stream(stream))


def bastion_accept_workspace_size(B: int, n_max: int) -> int:
    return int(lib().bastion_accept_workspace_size(B, n_max))


def bastion_accept(target, n, parent, token, K: int, acc_len, acc_nodes, acc_tok, bonus, ws, argmax_out=None,
                   dev_err=None, stream=None) -> None:
    """Stage 4. target [B, n_max, V] f32/bf16 with contiguous rows."""
    B, N, V = target.shape
    if target.stride(-1) != 1 or target.stride(0) != N * target.stride(1):
        raise BastionError("target must be [B, n_max, V] with a uniform row stride")
    row_stride = target.stride(1)
    _need(n, torch.int32, (B,), "n")
    _need(parent, torch.int32, (B, N), "parent")
    _need(token, torch.int32, (B, N), "token")
    _need(acc_len, torch.int32, (B,), "acc_len")
    _need(acc_nodes, torch.int32, (B, K + 1), "acc_nodes")
    _need(acc_tok, torch.int32, (B, K + 1), "acc_tok")
    _need(bonus, torch.int32, (B,), "bonus")
    _need(ws, torch.uint8, None, "ws")
    if argmax_out is not None:
        _need(argmax_out, torch.int32, (B, N), "argmax_out")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    _call("bastion_accept", _ptr(target), _dtype_code(target), B, N, V, row_stride, int(K), _ptr(n), _ptr(parent),
          _ptr(token), _ptr(acc_len), _ptr(acc_nodes), _ptr(acc_tok), _ptr(bonus), _ptr(argmax_out), _ptr(ws),
          ws.numel(), _ptr(dev_err), _stream(stream))


def bastion_accept_noalloc(target, n, parent, token, K: int, acc_len, acc_nodes, acc_tok, bonus, argmax_out=None,
                           dev_err=None, stream=None) -> None:
    """Stage 4 without a workspace, for callers that cannot allocate device
    memory at step time; the scratch is a fixed array inside the library
    (calls must not overlap on the GPU).  Same arguments as bastion_accept
    minus ``ws``."""
    B, N, V = target.shape
    if target.stride(-1) != 1 or target.stride(0) != N * target.stride(1):
        raise BastionError("target must be [B, n_max, V] with a uniform row stride")
    _need(n, torch.int32, (B,), "n")
    _need(parent, torch.int32, (B, N), "parent")
    _need(token, torch.int32, (B, N), "token")
    _need(acc_len, torch.int32, (B,), "acc_len")
    _need(acc_nodes, torch.int32, (B, K + 1), "acc_nodes")
    _need(acc_tok, torch.int32, (B, K + 1), "acc_tok")
    _need(bonus, torch.int32, (B,), "bonus")
    if argmax_out is not None:
        _need(argmax_out, torch.int32, (B, N), "argmax_out")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    _check(lib().bastion_accept_noalloc(_ptr(target), _dtype_code(target), B, N, V, target.stride(1), int(K),
                                        _ptr(n), _ptr(parent), _ptr(token), _ptr(acc_len), _ptr(acc_nodes),
                                        _ptr(acc_tok), _ptr(bonus), _ptr(argmax_out), _ptr(dev_err),
                                        _stream(stream)), "bastion_accept_noalloc")


def bastion_kv_commit(k_tree, v_tree, kv: "KV", acc_len, acc_nodes, ctx_len, ctx_out, dev_err=None,
                      stream=None) -> None:
    """After acceptance: append each request's accepted path (acc_nodes, root
    first, acc_len + 1 nodes) to the context cache at positions ctx_len ..
    ctx_len + acc_len and set ctx_out = ctx_len + acc_len + 1 (ctx_out may be
    ctx_len).  k_tree/v_tree [B, n_max, Hkv, d] (the cache's dtype);
    acc_nodes int32 [B, K+1]; acc_len, ctx_len, ctx_out int32 [B].  kv's k and v
    are written."""
    B, N, Hkv, d = k_tree.shape
    dt = k_tree.dtype
    _need(k_tree, dt, None, "k_tree")
    _need(v_tree, dt, (B, N, Hkv, d), "v_tree")
    _need(kv.k, dt, None, "kv.k")
    _need(kv.v, dt, tuple(kv.k.shape), "kv.v")
    if kv.block_table is not None:
        _need(kv.block_table, torch.int32, None, "block_table")
    _need(acc_len, torch.int32, (B,), "acc_len")
    if acc_nodes.dim() != 2 or acc_nodes.shape[0] != B:
        raise BastionError("acc_nodes must be [B, K+1]")
    _need(acc_nodes, torch.int32, None, "acc_nodes")
    K = acc_nodes.shape[1] - 1
    _need(ctx_len, torch.int32, (B,), "ctx_len")
    _need(ctx_out, torch.int32, (B,), "ctx_out")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    s = kv.c_struct()
    _check(lib().bastion_kv_commit(_ptr(k_tree), _ptr(v_tree), _dtype_code(k_tree), B, N, Hkv, d, K, _ptr(acc_len),
                                   _ptr(acc_nodes), ctypes.byref(s), _ptr(ctx_len), _ptr(ctx_out), _ptr(dev_err),
                                   _stream(stream)), "bastion_kv_commit")


def bastion_block_mask(n, block: int, mask, dev_err=None, stream=None) -> None:
    """Block-diffusion drafter mask for bastion_tree_attn: mask int64
    [B, n_max, ceil(n_max/64)] gets, for row i < n[b], the bits j < n[b] with
    i // block == j // block; n int32 [B]."""
    B = n.shape[0]
    _need(n, torch.int32, (B,), "n")
    if mask.dim() != 3 or mask.shape[0] != B:
        raise BastionError("mask must be [B, n_max, ceil(n_max/64)]")
    N = mask.shape[1]
    _need(mask, torch.int64, (B, N, (N + 63) // 64), "mask")
    if dev_err is not None:
        _need(dev_err, torch.int32, (1,), "dev_err")
    _check(lib().bastion_block_mask(B, N, int(block), _ptr(n), _ptr(mask), _ptr(dev_err), _stream(stream)),
           "bastion_block_mask")


def bastion_fit_verify_latency(N, t_us, knee_lo: int, knee_hi: int):
    """Host fit of T_verify(N) = a + b N + c max(0, N - knee) to measured times
    (sequences of equal length, at least two distinct N).  Returns
    (a, b, c, knee, sse)."""
    import numpy as np
    N = np.ascontiguousarray(N, dtype=np.int32)
    t = np.ascontiguousarray(t_us, dtype=np.float64)
    if N.shape != t.shape or N.ndim != 1:
        raise BastionError("N and t must be 1-D and of equal length")
    abc = np.zeros(3, dtype=np.float64)
    knee = ctypes.c_int32(0)
    sse = ctypes.c_double(0.0)
    _check(lib().bastion_fit_verify_latency(N.ctypes.data, t.ctypes.data, int(N.size), int(knee_lo), int(knee_hi),
                                            abc.ctypes.data, ctypes.byref(knee), ctypes.byref(sse)),
           "bastion_fit_verify_latency")
    return float(abc[0]), float(abc[1]), float(abc[2]), int(knee.value), float(sse.value)


def bastion_latency_table(a: float, b: float, c: float, knee: int, t_draft: float, n_max: int):
    """The stage-2 table C[0..n_max] (numpy float32, to be copied to the
    device) and L_AR = T_verify(1)."""
    import numpy as np
    abc = np.array([a, b, c], dtype=np.float64)
    C = np.zeros(n_max + 1, dtype=np.float32)
    L_AR = ctypes.c_float(0.0)
    _check(lib().bastion_latency_table(abc.ctypes.data, int(knee), float(t_draft), int(n_max), C.ctypes.data,
                                       ctypes.byref(L_AR)), "bastion_latency_table")
    return C, float(L_AR.value)


# --------------------------------------------------------------------------
# the whole step: buffers + the four calls
# --------------------------------------------------------------------------


class SpecTreeStep:
    """Owns the output buffers and workspaces of one spec-tree step and runs the
    four library calls in order on the current stream (no host sync inside)."""

    def __init__(self, B: int, K: int, V: int, topk: int, n_min: int, n_max: int, Hq: int, Hkv: int, d: int,
                 kv: KV, device="cuda", act_dtype=torch.bfloat16):
        self.B, self.K, self.V, self.topk = B, K, V, topk
        self.n_min, self.n_max, self.Hq, self.Hkv, self.d = n_min, n_max, Hq, Hkv, d
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.ids = torch.empty(B, K, topk, **i32)
        self.lg = torch.empty(B, K, topk, **f32)
        self.q = torch.empty(B, K, topk, **f32)
        self.lse = torch.empty(B, K, dtype=torch.float64, device=dev)
        W = (n_max + 63) // 64
        # n, acc_len, bonus and acc_tok share one block, so that a step's
        # result comes back to the host in a single copy
        self.result = torch.empty(3 * B + B * (K + 1), **i32)
        self.n = self.result[0:B]
        self.acc_len = self.result[B:2 * B]
        self.bonus = self.result[2 * B:3 * B]
        self.acc_tok = self.result[3 * B:].view(B, K + 1)
        self.parent = torch.empty(B, n_max, **i32)
        self.token = torch.empty(B, n_max, **i32)
        self.depth = torch.empty(B, n_max, **i32)
        self.pos = torch.empty(B, n_max, **i32)
        self.rho = torch.empty(B, n_max, **f32)
        self.mask = torch.empty(B, n_max, W, dtype=torch.int64, device=dev)
        self.ahat = torch.empty(B, **f32)
        self.S = torch.empty(B, **f32)
        self.S_curve = torch.empty(B, n_max, **f32)
        self.attn_out = torch.empty(B, n_max, Hq, d, dtype=act_dtype, device=dev)
        self.acc_nodes = torch.empty(B, K + 1, **i32)
        self.argmax = torch.empty(B, n_max, **i32)
        self.dev_err = torch.zeros(1, **i32)
        self.attn_ws = torch.zeros(max(1, bastion_tree_attn_workspace_size(B, n_max, Hq, Hkv, d, kv)),
                                   dtype=torch.uint8, device=dev)
        self.acc_ws = torch.zeros(bastion_accept_workspace_size(B, n_max), dtype=torch.uint8, device=dev)

    def draft(self, logits, root_tok, ctx_len, C, L_AR, stream=None):
        bastion_topk_softmax(logits, self.topk, self.ids, self.lg, self.q, self.lse, dev_err=self.dev_err,
                             stream=stream)
        bastion_tree_build(self.ids, self.lg, self.lse, self.V, root_tok, ctx_len, self.n_min, self.n_max, C, L_AR,
                           self.n, self.parent, self.token, self.depth, self.pos, self.rho, self.mask, self.ahat,
                           self.S, self.S_curve, dev_err=self.dev_err, stream=stream)

    def verify(self, q, k_tree, v_tree, kv: KV, ctx_len, scale, target, stream=None):
        bastion_tree_attn(q, k_tree, v_tree, kv, ctx_len, self.mask, self.n, self.attn_out, scale, ws=self.attn_ws,
                          dev_err=self.dev_err, stream=stream)
        bastion_accept(target, self.n, self.parent, self.token, self.K, self.acc_len, self.acc_nodes, self.acc_tok,
                       self.bonus, self.acc_ws, argmax_out=self.argmax, dev_err=self.dev_err, stream=stream)

    def __call__(self, logits, root_tok, ctx_len, C, L_AR, q, k_tree, v_tree, kv: KV, scale, target, stream=None):
        self.draft(logits, root_tok, ctx_len, C, L_AR, stream=stream)
        self.verify(q, k_tree, v_tree, kv, ctx_len, scale, target, stream=stream)

    def prepare(self, logits, root_tok, ctx_len, C, L_AR, q, k_tree, v_tree, kv: KV, scale, target,
                stream=None) -> "PreparedStep":
        """Check and marshal the four calls of a step on these inputs once,
        without launching anything; the returned object issues them on each
        call.  Its stream is fixed now (``stream``, else the current one), and
        it keeps the input tensors alive, whose contents may change between
        calls but whose storage must not."""
        if getattr(_rec, "calls", None) is not None:
            raise BastionError("prepare() does not nest")
        _rec.calls = []
        try:
            self(logits, root_tok, ctx_len, C, L_AR, q, k_tree, v_tree, kv, scale, target, stream=stream)
            calls = _rec.calls
        finally:
            _rec.calls = None
        return PreparedStep(calls, (self, logits, root_tok, ctx_len, C, q, k_tree, v_tree, kv, target))


class PreparedStep:
    """The four library calls of one spec-tree step with their arguments
    already checked and marshalled (see ``SpecTreeStep.prepare``): calling it
    only crosses the C ABI four times."""

    def __init__(self, calls, keep):
        self._calls = tuple(calls)
        self._keep = keep   # the tensors whose device pointers the calls hold

    def __call__(self) -> None:
        for fn, args, name in self._calls:
            _check(fn(*args), name)


class HostStepRunner:
    """Spec-tree steps whose per-step inputs come from pinned host memory.

    Each of ``depth`` slots owns a pinned host block and a device block that
    hold the step's drafter logits, root tokens, context lengths, tree Q/K/V
    and target logits back to back (each 256-byte aligned), plus a pinned
    result block.  The caller fills ``inputs(slot)`` (views of the host block)
    and calls ``submit()``: the host block goes to the device in ``copy_split``
    equal pieces, each a single copy on its own copy stream (several copy
    engines in parallel), the step (a CUDA graph of the four library calls, captured
    once per slot) runs on the compute stream when that copy has landed, and
    the result block (n, acc_len, bonus, acc_tok) comes back in one copy.  The
    copy of the next slot overlaps the step in flight.  ``collect()`` waits
    for the oldest submitted step and returns its result views.

    The context KV cache, the latency table ``C``, ``L_AR`` and the softmax
    scale are model state: they stay on the device and are fixed per runner.
    """

    _ALIGN = 256

    def __init__(self, step: SpecTreeStep, kv: KV, C: Optional[torch.Tensor], L_AR: float, scale: float,
                 act_dtype=torch.bfloat16, depth: int = 2, copy_split: int = 1):
        if depth < 1:
            raise BastionError("depth must be >= 1")
        st = step
        B, K, V, N, Hq, Hkv, d = st.B, st.K, st.V, st.n_max, st.Hq, st.Hkv, st.d
        self.step, self.kv, self.C, self.L_AR, self.scale = step, kv, C, float(L_AR), float(scale)
        self.fields = (("logits", (B, K, V), act_dtype), ("root_tok", (B,), torch.int32),
                       ("ctx_len", (B,), torch.int32), ("q", (B, N, Hq, d), act_dtype),
                       ("k_tree", (B, N, Hkv, d), act_dtype), ("v_tree", (B, N, Hkv, d), act_dtype),
                       ("target", (B, N, V), act_dtype))
        self.offsets = {}
        off = 0
        for name, shape, dt in self.fields:
            off = (off + self._ALIGN - 1) // self._ALIGN * self._ALIGN
            self.offsets[name] = off
            nbytes = torch.Size(shape).numel() * torch.empty(0, dtype=dt).element_size()
            off += nbytes
        self.block_bytes = off
        self.result_numel = st.result.numel()
        self.depth = depth
        dev = st.result.device
        # zero-filled, so that the run made while capturing a slot's graph
        # reads valid inputs (all-equal logits, empty contexts)
        self.host = [torch.zeros(off, dtype=torch.uint8, pin_memory=True) for _ in range(depth)]
        self.dev = [torch.zeros(off, dtype=torch.uint8, device=dev) for _ in range(depth)]
        self.res_host = [torch.empty(self.result_numel, dtype=torch.int32, pin_memory=True) for _ in range(depth)]
        self.copy_streams = [torch.cuda.Stream(device=dev) for _ in range(max(1, copy_split))]
        n = len(self.copy_streams)
        piece = (off + n - 1) // n
        piece = (piece + self._ALIGN - 1) // self._ALIGN * self._ALIGN
        self.pieces = [(a, min(off, a + piece)) for a in range(0, off, piece)]
        self.stream = torch.cuda.Stream(device=dev)
        self.copied = [[torch.cuda.Event() for _ in self.pieces] for _ in range(depth)]
        self.consumed = [torch.cuda.Event() for _ in range(depth)]
        self.done = [torch.cuda.Event() for _ in range(depth)]
        self.graphs = [None] * depth
        self.in_flight = []   # slots submitted and not yet collected, oldest first
        self.next_slot = 0

    @property
    def h2d_bytes(self) -> int:
        return self.block_bytes

    @property
    def d2h_bytes(self) -> int:
        return self.result_numel * 4

    def _views(self, block: torch.Tensor) -> dict:
        out = {}
        for name, shape, dt in self.fields:
            o = self.offsets[name]
            nbytes = torch.Size(shape).numel() * torch.empty(0, dtype=dt).element_size()
            out[name] = block[o:o + nbytes].view(dt).view(shape)
        return out

    def inputs(self, slot: int) -> dict:
        """Pinned host views of slot ``slot``'s inputs, to be filled by the caller."""
        return self._views(self.host[slot])

    def _run(self, slot: int) -> None:
        v = self._views(self.dev[slot])
        self.step(v["logits"], v["root_tok"], v["ctx_len"], self.C, self.L_AR, v["q"], v["k_tree"], v["v_tree"],
                  self.kv, self.scale, v["target"], stream=self.stream)

    def _graph(self, slot: int) -> torch.cuda.CUDAGraph:
        if self.graphs[slot] is None:
            torch.cuda.synchronize()
            with torch.cuda.stream(self.stream):
                self._run(slot)   # first call outside capture: lazy set-up in the library
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self._run(slot)
            torch.cuda.synchronize()
            self.graphs[slot] = g
        return self.graphs[slot]

    def prepare(self) -> None:
        """Capture every slot's graph now (otherwise the first submit does)."""
        for slot in range(self.depth):
            self._graph(slot)

    def submit(self) -> int:
        """Start the step of the next slot; returns the slot.  Waits for the
        oldest step first when all slots are in flight."""
        if len(self.in_flight) == self.depth:
            self.collect()
        slot = self.next_slot
        self.next_slot = (slot + 1) % self.depth
        g = self._graph(slot)
        st = self.stream
        for (a, b), cs, ev in zip(self.pieces, self.copy_streams, self.copied[slot]):
            cs.wait_event(self.consumed[slot])   # the step that last read this device block has finished
            with torch.cuda.stream(cs):
                self.dev[slot][a:b].copy_(self.host[slot][a:b], non_blocking=True)
                ev.record(cs)
        for ev in self.copied[slot]:
            st.wait_event(ev)
        with torch.cuda.stream(st):
            g.replay()
            self.consumed[slot].record(st)
            self.res_host[slot].copy_(self.step.result, non_blocking=True)
            self.done[slot].record(st)
        self.in_flight.append(slot)
        return slot

    def collect(self) -> dict:
        """Wait for the oldest step in flight; its n, acc_len, bonus, acc_tok (host views)."""
        if not self.in_flight:
            raise BastionError("no step in flight")
        slot = self.in_flight.pop(0)
        self.done[slot].synchronize()
        r = self.res_host[slot]
        B, K = self.step.B, self.step.K
        return {"n": r[0:B], "acc_len": r[B:2 * B], "bonus": r[2 * B:3 * B], "acc_tok": r[3 * B:].view(B, K + 1)}
