"""Shared test helpers: run the oracle over a synthetic workload.

Only the oracle side lives here (the CUDA side is driven through the package's
binding in the GPU tests).  Both sides start from the same synthetic inputs of
``synth`` and each builds its own page pool with its own append.
"""
from __future__ import annotations

import numpy as np

import oracle
from synth import SENTINEL_BF16


def oracle_pool(wl):
    """Sentinel-filled pool holding every sequence's initially cached prefix."""
    pool = oracle.new_pool(wl.pool_shape(), SENTINEL_BF16)
    t = wl.initial_table()
    k, v = wl.initial_kv()
    oracle.kv_append(pool, k, v, t["qo_indptr"], t["page_indices"], t["kv_indptr"], t["last_page_len"])
    return pool


def oracle_step(wl, pool, k, sel_rows=None, tree_mask=None):
    """Append step k's new K/V into `pool` (in place) and attend: (out, lse, pairs).
    A step with draft trees attends under its tree mask (or `tree_mask`)."""
    t = wl.step_table(k)
    q, kn, vn = wl.step_inputs(k)
    oracle.kv_append(pool, kn, vn, t["qo_indptr"], t["page_indices"], t["kv_indptr"], t["last_page_len"])
    if tree_mask is None and wl.has_tree(k):
        tree_mask = wl.tree_mask(k)
    return oracle.attention(q, pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"],
                            t["last_page_len"], wl.causal, wl.sm_scale, wl.num_qo_heads,
                            sel_rows=sel_rows, tree_mask=tree_mask)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 (round to nearest even, via fp32) -> fp64, for error reporting."""
    import torch
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16).double().numpy()


def err_stats(gpu: np.ndarray, ref: np.ndarray):
    """max |err|, mean |err|, relative L2 of gpu (fp64 view of bf16) vs ref."""
    d = np.abs(gpu.astype(np.float64) - ref)
    rel = float(np.linalg.norm(gpu.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300))
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0, rel
