"""Drive the CUDA path over a synthetic workload (GPU tests and smoke only)."""
from __future__ import annotations

import copy

import numpy as np
import torch

import decode_attention_append_gb300 as daa
from synth import SENTINEL_BF16


def new_pool(wl, device):
    return torch.full(wl.pool_shape(), SENTINEL_BF16, dtype=torch.int16, device=device).view(torch.bfloat16)


def gpu_fill(wl, pool, device):
    """Append every sequence's initially cached prefix (the CUDA append)."""
    it = wl.initial_table()
    k0, v0 = wl.initial_kv()
    if k0.shape[0] == 0:
        return
    t = daa.PageTable.from_host(it["qo_indptr"], it["kv_indptr"], it["page_indices"],
                                it["last_page_len"], device)
    daa.kv_append(k0.to(device), v0.to(device), pool, t.qo_indptr, t.page_indices, t.kv_indptr,
                  t.last_page_len)


def gpu_step(wl, pool, k, device, with_lse=True, fused=False, groups=False):
    """Append step k's new K/V and run attention: (out bf16 cpu, lse fp32 cpu).
    fused: one append_attention call instead of kv_append + batch_attention.
    groups: pass the step's prefix groups (the shared-prefix calls).
    A step with draft trees appends, then attends under its tree mask."""
    st = wl.step_table(k)
    q, kn, vn = wl.step_inputs(k)
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                  st["last_page_len"], device)
    runner = daa.BatchAttention(tab, wl.num_qo_heads, pool, causal=wl.causal, sm_scale=wl.sm_scale,
                                prefix_groups=wl.prefix_groups(k) if groups else None)
    qd = q.to(device)
    lse = torch.full((q.shape[0], wl.num_qo_heads), float("nan"), device=device) if with_lse else None
    out = torch.full_like(qd, float("nan"))
    if wl.has_tree(k):
        mask = torch.from_numpy(wl.tree_mask(k).view(np.int32)).to(device)
        if kn.shape[0]:
            runner.append(kn.to(device), vn.to(device))
        runner.run(qd, out=out, lse=lse, tree_mask=mask)
    elif fused:
        runner.step(kn.to(device), vn.to(device), qd, out=out, lse=lse)
    else:
        if kn.shape[0]:
            runner.append(kn.to(device), vn.to(device))
        runner.run(qd, out=out, lse=lse)
    torch.cuda.synchronize()
    return out.cpu(), (lse.cpu() if lse is not None else None)


def pool_bits(pool: torch.Tensor) -> np.ndarray:
    return pool.view(torch.int16).cpu().numpy().view(np.uint16)


def compact(wl):
    """Copy of wl whose pages are renumbered 0..n-1 in order of first use (so
    the oracle's pool holds only the pages the workload touches; a page shared
    by several sequences stays shared)."""
    w = copy.copy(wl)
    w.seqs = []
    mapping = {}
    for s in wl.seqs:
        for a in s.pages:
            mapping.setdefault(int(a), len(mapping))
        new = np.asarray([mapping[int(a)] for a in s.pages], np.int32)
        w.seqs.append(type(s)(s.length, new, s.prefix, s.prefix_len))
    w.num_pages = max(1, len(mapping))
    return w, mapping
