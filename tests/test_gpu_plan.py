"""Plan once, run many (daa_batch_attention_plan / _run / daa_append_attention_run):
runs on a stored plan give the bits of the calls that plan for themselves,
run after run, with and without prefix groups and with the fused append."""
import numpy as np
import pytest
import torch

from synth import make_prefix_groups_workload, make_random_workload, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _setup(wl, dev, groups):
    import decode_attention_append_gb300 as daa
    from gpu_support import gpu_fill, new_pool
    pool = new_pool(wl, dev)
    gpu_fill(wl, pool, dev)
    st = wl.step_table(0)
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                  st["last_page_len"], dev)
    pg = wl.prefix_groups(0) if groups else None
    runner = daa.BatchAttention(tab, wl.num_qo_heads, pool, causal=wl.causal, sm_scale=wl.sm_scale,
                                prefix_groups=pg)
    return daa, pool, tab, runner


CASES = [
    ("mixed", lambda: make_random_workload(
        501, 32, 8, 128, 16, [(300, 1500), (1, 4000), (7, 900), (40, 2000), (1, 77), (1, 9000)],
        extra_pages=9), False),
    ("mha_d64", lambda: make_random_workload(502, 8, 8, 64, 16, [(1, 3000), (1, 129), (100, 800)],
                                             extra_pages=5), False),
    ("groups", lambda: make_prefix_groups_workload(
        "g503", 32, 8, 128, 16, 503, [("group", 1024, [(1, 1100 + 97 * i) for i in range(10)] + [(9, 2000)])]),
     True),
    ("gqa_shard", lambda: make_workload("gqa_decode_shard"), False),
]


@pytest.mark.parametrize("name,make,groups", CASES, ids=[c[0] for c in CASES])
def test_runs_on_a_plan_match_planning_calls(dev, name, make, groups):
    wl = make()
    daa, pool, tab, runner = _setup(wl, dev, groups)
    q0, kn, vn = wl.step_inputs(0)
    runner.append(kn.to(dev), vn.to(dev))
    g = torch.Generator().manual_seed(7)
    qs = [q0.to(dev)] + [torch.randn(q0.shape, generator=g).to(torch.bfloat16).to(dev) for _ in range(2)]
    ref = []
    for q in qs:  # each call plans for itself
        lse = torch.empty(q.shape[0], wl.num_qo_heads, device=dev)
        ref.append((runner.run(q, lse=lse), lse))
    runner.plan()
    for rep in range(2):  # the same plan, run after run
        for q, (o_ref, l_ref) in zip(qs, ref):
            lse = torch.empty_like(l_ref)
            out = runner.run(q, lse=lse)
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), o_ref.view(torch.int16)), (name, rep)
            assert torch.equal(lse, l_ref), (name, rep)
    assert daa.device_error(reset=True) == 0


@pytest.mark.parametrize("groups,fusion_at_run", [(False, True), (True, True), (False, False)])
def test_append_attention_run_matches_fused_call(dev, groups, fusion_at_run):
    """A fused run on a stored plan gives the bits of the fused call that plans
    for itself, also when the prefill append fusion is switched off between the
    plan and the run (the run's append then covers every row)."""
    wl = make_prefix_groups_workload("g504", 32, 8, 128, 16, 504,
                                     [("group", 512, [(1, 600 + 131 * i) for i in range(12)]),
                                      ("solo", 200, 700), ("solo", 1, 3000)])
    q, kn, vn = (x.to(dev) for x in wl.step_inputs(0))
    outs, pools = [], []
    for planned in (False, True):
        daa, pool, tab, runner = _setup(wl, dev, groups)
        if planned:
            runner.plan()
        lse = torch.empty(q.shape[0], wl.num_qo_heads, device=dev)
        try:
            if planned and not fusion_at_run:
                daa.set_prefill_append_fusion(False)
            outs.append((runner.step(kn, vn, q, lse=lse), lse))
        finally:
            daa.set_prefill_append_fusion(True)
        pools.append(pool)
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(pools[0].view(torch.int16), pools[1].view(torch.int16))
