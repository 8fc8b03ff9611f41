"""Block-diffusion drafter attention: the mask builder (bit-exact against the
oracle) and the attention call driven by that mask (against the oracle's
mask-driven attention), contiguous and paged, bf16 and fp32."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import binding as bn  # noqa: E402
from tree_speculative_decoding_bastion_gb300 import inputs as I  # noqa: E402

from . import cases as C  # noqa: E402
from .test_gpu_parity import attn_tol  # noqa: E402

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_bastion_gb300 import build
    build.build()
    bn.bastion_init(0)


def gpu_mask(n, n_max, block):
    B = len(n)
    mask = torch.full((B, n_max, (n_max + 63) // 64), -1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_block_mask(C.dev(np.asarray(n, np.int32)), block, mask, dev_err=err)
    torch.cuda.synchronize()
    return mask.cpu().numpy().view(np.uint64), int(err.item())


@pytest.mark.parametrize("n,n_max,block", [([16, 16, 16, 16], 16, 16), ([64, 40, 1], 64, 16), ([256, 130], 256, 7),
                                           ([200, 3], 256, 64), ([50], 60, 300), ([17, 9], 20, 1)])
def test_block_mask_matches_oracle(n, n_max, block):
    got, err = gpu_mask(n, n_max, block)
    assert err == 0
    assert np.array_equal(got, oracle.block_mask(np.array(n), n_max, block))


def test_block_mask_bad_n_clears_the_request():
    got, err = gpu_mask([0, 12, 99], 64, 8)
    assert err & bn.DEVERR_N
    want = oracle.block_mask(np.array([0, 12, 0]), 64, 8)
    assert np.array_equal(got, want)


DRAFTERS = {
    # one block of 16 mask tokens per request after a 4096-token clean prefix
    "block16_b4": (W["qwen3_8b_b1"].scaled(name="drafter_b4", B=4, n_min=16, n_max=16, L=4096), 16, [16] * 4),
    # several isolated blocks, ragged, paged prefix
    "blocks_paged": (W["llama31_8b_b16_paged"].scaled(name="drafter_paged", B=3, n_min=64, n_max=64, L=3000,
                                                     L_min=200), 16, [64, 40, 23]),
    # fp32, blocks of 4
    "f32_block4": (W["tiny_v1024_f32"].scaled(name="drafter_f32", B=2, n_min=16, n_max=16, L=100), 4, [16, 11]),
}


@pytest.mark.parametrize("name", list(DRAFTERS))
def test_drafter_attention_matches_oracle(name):
    wl, block, n = DRAFTERS[name]
    inp = I.make_step_inputs(wl, 11)
    n = np.array(n, np.int32)
    kv = C.kv_of(inp)
    n_dev = C.dev(n)
    mask = torch.empty(wl.B, wl.n_max, (wl.n_max + 63) // 64, dtype=torch.int64, device="cuda")
    bn.bastion_block_mask(n_dev, block, mask)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    out = torch.full((wl.B, wl.n_max, wl.Hq, wl.d), float("nan"), device="cuda", dtype=dt)
    ws = torch.zeros(max(1, bn.bastion_tree_attn_workspace_size(wl.B, wl.n_max, wl.Hq, wl.Hkv, wl.d, kv)),
                     dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bn.bastion_tree_attn(C.dev(inp.q, wl.dtype), C.dev(inp.k_tree, wl.dtype), C.dev(inp.v_tree, wl.dtype), kv,
                         C.dev(inp.ctx_len), mask, n_dev, out, inp.scale, ws=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.float().cpu().numpy()
    m = oracle.block_mask(n, wl.n_max, block)
    assert np.array_equal(mask.cpu().numpy().view(np.uint64), m)
    rng = np.random.default_rng(0)
    rows = sorted({(b, int(i), int(h)) for b in range(wl.B)
                   for i, h in zip(rng.integers(0, n[b], 12), rng.integers(0, wl.Hq, 12))}
                  | {(b, int(n[b]) - 1, wl.Hq - 1) for b in range(wl.B)})
    f = lambda a: I.as_f32(a, wl.dtype)
    want = oracle.masked_attention(f(inp.q), f(inp.k_tree), f(inp.v_tree), f(inp.k_ctx), f(inp.v_ctx), inp.ctx_len,
                                   m, n, wl.Hkv, inp.scale, block_table=inp.block_table, page_size=wl.page_size,
                                   rows=rows)
    atol, rtol = attn_tol(wl)
    for r in rows:
        assert np.all(np.abs(got[r] - want[r]) <= atol + rtol * np.abs(want[r])), r
    for b in range(wl.B):
        assert np.isnan(got[b, int(n[b]):]).all()
