"""daa_batch_attention_noalloc, the entry point for callers that cannot allocate
device memory (a serving engine whose HBM all belongs to its page pool, a
latency-critical path where cudaMalloc could synchronise the device, a
foreign-language host without a CUDA allocator).  Its scratch is the library's
fixed device array instead of a caller workspace.

Checked through the C ABI, on two calls in a row with different batches (so
the second call runs over the first call's leftover scratch contents):
* against daa_batch_attention (the workspace entry point): both build the same
  plan and run the same kernels, so out and lse must be bit-identical;
* against the CPU oracle at the parity tolerances of the other GPU tests;
* a batch past the scratch array's unit limit is rejected with
  DAA_ERR_WORKSPACE before anything is enqueued (out stays untouched).
This file is collected last and is self-contained: it passes alone in a fresh
process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import make_random_workload

pytestmark = pytest.mark.gpu

MAX_ERR, MEAN_ERR, REL_L2, LSE_ERR = 1.5e-2, 2e-3, 1e-2, 1e-3
DAA_ERR_WORKSPACE = -6


def _setup(wl, dev):
    from gpu_support import gpu_fill, new_pool
    import decode_attention_append_gb300 as daa
    pool = new_pool(wl, dev)
    gpu_fill(wl, pool, dev)
    st = wl.step_table(0)
    q, kn, vn = wl.step_inputs(0)
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                  st["last_page_len"], dev)
    daa.kv_append(kn.to(dev), vn.to(dev), pool, tab.qo_indptr, tab.page_indices, tab.kv_indptr,
                  tab.last_page_len)
    return pool, tab, q.to(dev)


def _dims(wl):
    import decode_attention_append_gb300 as daa
    return daa._Dims(wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages)


def _call_noalloc(lib, wl, pool, tab, q, out, lse):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    h = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    return lib.daa_batch_attention_noalloc(
        p(q), p(pool), p(tab.qo_indptr), p(tab.kv_indptr), p(tab.page_indices), p(tab.last_page_len),
        h(tab.h_qo_indptr), h(tab.h_kv_indptr), h(tab.h_last_page_len), len(tab.h_qo_indptr) - 1,
        1, ctypes.c_float(wl.sm_scale), p(out), p(lse), _dims(wl),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _call_workspace(lib, wl, pool, tab, q, out, lse):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    h = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    dims = _dims(wl)
    status = ctypes.c_int32(0)
    nbytes = lib.daa_batch_attention_workspace_size(h(tab.h_qo_indptr), h(tab.h_kv_indptr),
                                                    h(tab.h_last_page_len), len(tab.h_qo_indptr) - 1,
                                                    dims, ctypes.byref(status))
    assert status.value == 0
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.daa_batch_attention(
        p(q), p(pool), p(tab.qo_indptr), p(tab.kv_indptr), p(tab.page_indices), p(tab.last_page_len),
        h(tab.h_qo_indptr), h(tab.h_kv_indptr), h(tab.h_last_page_len), len(tab.h_qo_indptr) - 1,
        1, ctypes.c_float(wl.sm_scale), p(out), p(lse), p(ws), ctypes.c_size_t(ws.numel()), dims,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.daa_status_string(st)
    torch.cuda.synchronize()  # the workspace is freed on return
    return nbytes


def _oracle(wl):
    from gpu_support import compact
    from support import oracle_pool, oracle_step
    cw, _ = compact(wl)
    pool = oracle_pool(cw)
    ref, ref_lse, _ = oracle_step(cw, pool, 0)
    return ref, ref_lse


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import decode_attention_append_gb300 as daa
    return daa.load_library()


def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(lib):
    import decode_attention_append_gb300 as daa
    from support import err_stats
    dev = torch.device("cuda:0")
    batches = [
        # mixed: a prefill chunk, long decodes that are split (partials + merge), short decodes
        make_random_workload(301, 8, 2, 128, 16, [(200, 1200), (1, 40000), (1, 300), (1, 9000)]),
        # a different shape on the second call: GQA 4:1, d 64, more splits
        make_random_workload(302, 8, 2, 64, 16, [(1, 30000), (37, 37), (1, 17), (1, 25000)]),
    ]
    for wl in batches:
        pool, tab, q = _setup(wl, dev)
        out_ref = torch.full_like(q, float("nan"))
        lse_ref = torch.full((q.shape[0], wl.num_qo_heads), float("nan"), device=dev)
        nbytes = _call_workspace(lib, wl, pool, tab, q, out_ref, lse_ref)
        assert nbytes > 0
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = _call_noalloc(lib, wl, pool, tab, q, out, lse)
        assert st == 0, lib.daa_status_string(st)
        torch.cuda.synchronize()
        # same plan, same kernels: identical bits
        assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16)), wl.seed
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), wl.seed
        # and the method's result, against the fp64 oracle
        ref, ref_lse = _oracle(wl)
        got = out.cpu().double().numpy()
        assert np.isfinite(got).all()
        mx, mean, rel = err_stats(got, ref)
        assert mx <= MAX_ERR and mean <= MEAN_ERR and rel <= REL_L2, (wl.seed, mx, mean, rel)
        assert np.abs(lse.cpu().double().numpy() - ref_lse).max() <= LSE_ERR
    assert daa.device_error(reset=True) == 0


def test_noalloc_rejects_a_batch_past_its_unit_limit(lib):
    """16,385 one-token decode requests on one kv head give 16,385 decode splits,
    one more than the fixed plan buffers hold: DAA_ERR_WORKSPACE, nothing run."""
    import decode_attention_append_gb300 as daa
    dev = torch.device("cuda:0")
    n = 16385
    ar = np.arange(n + 1, dtype=np.int32)
    tab = daa.PageTable.from_host(ar, ar, ar[:n], np.ones(n, np.int32), dev)
    pool = torch.zeros((n, 2, 1, 16, 64), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((n, 1, 64), dtype=torch.bfloat16, device=dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((n, 1), float("nan"), device=dev)

    class W:
        num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale = 1, 1, 64, 16, n, 0.125
    st = _call_noalloc(lib, W, pool, tab, q, out, lse)
    assert st == DAA_ERR_WORKSPACE, st
    torch.cuda.synchronize()
    assert bool(torch.isnan(out.float()).all()) and bool(torch.isnan(lse).all())
    assert daa.device_error(reset=True) == 0
