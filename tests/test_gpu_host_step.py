"""daa_append_attention_host: a serving step fed from pinned host memory (one
library call uploads the packed inputs, runs the fused append + attention and
reads the output back).  Its output must be exactly the fused call's on the
same inputs -- the same plan and kernels, only the copies are added -- for
several steps in a row over both device buffer sets, with the pool left
bit-identical; and the method's result against the oracle."""
import numpy as np
import pytest
import torch

from synth import make_random_workload
from support import err_stats, oracle_pool, oracle_step

pytestmark = pytest.mark.gpu

MAX_ERR, MEAN_ERR, REL_L2 = 1.5e-2, 2e-3, 1e-2

CASES = [
    # (seed, Hq, Hkv, d, [(qo, kv), ...]): a chunk on the pair kernel, split
    # decodes, a short request; GQA 4:1 head_dim 128 and MHA head_dim 64
    (151, 32, 8, 128, [(300, 1000), (1, 5000), (1, 77), (40, 400)]),
    (152, 8, 8, 64, [(200, 700), (1, 3000), (1, 16), (9, 9)]),
]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_host_step_matches_fused_call(dev, case):
    import decode_attention_append_gb300 as daa
    from gpu_support import compact, gpu_fill, gpu_step, new_pool, pool_bits
    seed, Hq, Hkv, d, reqs = case
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=5)
    # reference: the fused call on device tensors
    pa = new_pool(wl, dev)
    gpu_fill(wl, pa, dev)
    ref_out, _ = gpu_step(wl, pa, 0, dev, fused=True)
    # host steps: three in a row (buffer sets 0, 1, 0), same step inputs
    pb = new_pool(wl, dev)
    gpu_fill(wl, pb, dev)
    st = wl.step_table(0)
    q, kn, vn = wl.step_inputs(0)
    sections = {n: torch.from_numpy(st[n]) for n in ("qo_indptr", "kv_indptr", "page_indices",
                                                     "last_page_len")}
    sections.update(q=q, k_new=kn, v_new=vn)
    hs = daa.HostStep(sections, pb, Hq, causal=True, sm_scale=wl.sm_scale)
    for i in range(3):
        hs.step(i)
    for i in range(3):
        hs.done(i).synchronize()
        if i < 2:
            got = hs.out(i).clone()
            assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16)), f"step {i}"
    torch.cuda.synchronize()
    assert torch.equal(hs.out(2).view(torch.int16), ref_out.view(torch.int16))
    assert np.array_equal(pool_bits(pa), pool_bits(pb))
    # against the oracle
    cw, _ = compact(wl)
    ref, _, _ = oracle_step(cw, oracle_pool(cw), 0)
    mx, mean, rel = err_stats(hs.out(2).double().numpy(), ref)
    assert mx <= MAX_ERR and mean <= MEAN_ERR and rel <= REL_L2, (mx, mean, rel)
    assert daa.device_error(reset=True) == 0
