"""CPU oracle of the spec-tree step: test infrastructure, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.
"""
from .bastion_oracle import (  # noqa: F401
    Tree,
    accept,
    attend,
    block_mask,
    context_kv,
    fit_verify_latency,
    kv_commit,
    latency_table,
    marginals,
    masked_attention,
    path_to_root,
    stack_trees,
    topk_softmax,
    tree_attention,
    tree_build,
)
