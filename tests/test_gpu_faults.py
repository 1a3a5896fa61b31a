"""Failure detection on the GPU without a GPU fault.

* A page id outside the pool (page ids are only on the device, so the host
  cannot check them) is caught by the kernels' own bounds checks on every
  route -- append, CUDA-core decode, tensor-core decode and verify items, short
  items, pair prefill, single-CTA prefill -- and recorded in the device error
  word (code 1); the call's outputs are undefined but nothing outside the
  given buffers is touched and the context stays usable.
* The bounded wait every kernel uses gives up after its time limit on a
  barrier nothing completes (code 2), and the kernel exits.
After each, a valid call matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from synth import SENTINEL_BF16, make_random_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


ROUTES = [
    # (seed, Hq, Hkv, d, [(qo, kv), ...], request whose page is corrupted, what runs it)
    (401, 8, 8, 128, [(1, 700), (1, 40)], 0, "CUDA-core decode"),
    (402, 32, 4, 128, [(1, 900), (5, 300)], 0, "tensor-core decode"),
    (403, 32, 4, 128, [(1, 900), (5, 300)], 1, "tensor-core verify item"),
    (404, 32, 8, 128, [(40, 500), (1, 100)], 0, "short item"),
    (405, 32, 8, 128, [(300, 700)], 0, "pair prefill"),
    (406, 16, 4, 64, [(200, 450)], 0, "single-CTA prefill"),
]


@pytest.mark.parametrize("case", ROUTES, ids=lambda c: c[6].replace(" ", "_"))
@pytest.mark.parametrize("bad", ["past_end", "negative"])
def test_page_id_out_of_range_is_recorded(dev, case, bad):
    import decode_attention_append_gb300 as daa
    from gpu_support import gpu_fill, new_pool, pool_bits
    seed, Hq, Hkv, d, reqs, r_bad, _ = case
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=3)
    pool = new_pool(wl, dev)
    gpu_fill(wl, pool, dev)
    assert daa.device_error(reset=True) == 0
    st = wl.step_table(0)
    q, kn, vn = wl.step_inputs(0)
    pages = st["page_indices"].copy()
    # corrupt the page holding the request's last (appended) token, so the
    # append, the last key split and the prefill's diagonal tile all meet it
    slot = st["kv_indptr"][r_bad + 1] - 1
    pages[slot] = wl.num_pages + 3 if bad == "past_end" else -5
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], pages, st["last_page_len"], dev)
    before = pool_bits(pool)
    runner = daa.BatchAttention(tab, Hq, pool, sm_scale=wl.sm_scale)
    runner.append(kn.to(dev), vn.to(dev))
    torch.cuda.synchronize()
    assert daa.device_error(reset=False) == 1          # the append skipped the row
    after = pool_bits(pool)
    changed = np.flatnonzero((after != before).reshape(wl.num_pages, -1).any(axis=1))
    good_pages = set(int(p) for p in pages if 0 <= p < wl.num_pages)
    assert set(changed.tolist()) <= good_pages          # nothing written elsewhere
    runner.run(q.to(dev))
    torch.cuda.synchronize()
    assert daa.device_error(reset=True) == 1
    assert daa.device_error(reset=False) == 0


def test_bounded_wait_gives_up_and_context_survives(dev):
    import decode_attention_append_gb300 as daa
    assert daa.device_error(reset=True) == 0
    t0 = time.perf_counter()
    assert daa.selftest_bounded_wait()
    dt = time.perf_counter() - t0
    assert 0.5 < dt < 30.0, dt
    assert daa.device_error(reset=True) == 2
    assert daa.device_error(reset=False) == 0


def test_valid_call_after_recorded_errors_matches_oracle(dev):
    import decode_attention_append_gb300 as daa
    from test_gpu_parity import _run_both
    wl = make_random_workload(407, 32, 8, 128, 16, [(300, 700), (40, 500), (1, 900), (5, 300)],
                              extra_pages=3)
    _run_both(wl, dev)
    assert daa.device_error(reset=True) == 0
