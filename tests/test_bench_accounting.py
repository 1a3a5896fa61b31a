"""bench.py's algorithmic accounting on the named workloads (host only): the
bytes and FLOPs its rates and rooflines divide by follow the definitions they
state -- K/V read once per request, 4 d Hq FLOP per attended (query, key) pair
("Chunked prefill", #flops) -- and the append kernel's own bytes in a fused call
count only the rows the prefill kernels do not write themselves."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import make_workload  # noqa: E402


def _row_bytes(wl):
    return wl.num_kv_heads * wl.head_dim * 2 * 2 * 2  # K and V, read and written, bf16


def test_long_prompt_flops_match_the_causal_pair_count():
    wl = make_workload("long_prefill")
    acc = bench.step_accounting(wl)
    # 4 prompts, 8192 new over 8192 cached: each new token i sees 8192 + i + 1 keys
    L, c = 8192, 8192
    pairs = L * c + L * (L + 1) // 2
    assert acc["prefill_flops"] == 4 * 128 * 64 * pairs * 4


@pytest.mark.parametrize("name,fused_rows", [
    # every chunk's cached prefix is a multiple of 128 keys: only the decode rows remain
    ("long_prefill", 64),
    ("chunked_prefill_mixed", 32),
    ("prefix_shared", 64),
    ("long_prefill_d64", 32),
    ("first_chunk_prefill", 64),
    # decode only: every row
    ("mha_decode", 32),
    ("gqa_decode_shard", 128),
])
def test_append_kernel_bytes_in_a_fused_call(name, fused_rows):
    wl = make_workload(name)
    acc = bench.step_accounting(wl)
    assert acc["append_kernel_bytes_fused"] == fused_rows * _row_bytes(wl)
    assert acc["append_bytes"] == acc["nnz_new"] * _row_bytes(wl)


def test_tree_calls_append_every_row():
    wl = make_workload("tree_verify")
    acc = bench.step_accounting(wl)
    assert acc["append_kernel_bytes_fused"] == acc["append_bytes"]


def test_unaligned_prefix_leaves_the_mixed_tile_to_the_append():
    # a request whose cached prefix ends inside a 128-key tile: its new tokens
    # up to the next multiple of 128 go through the append kernel
    from synth import make_random_workload
    wl = make_random_workload(7, 32, 8, 128, 16, [(300, 1000), (1, 500)], extra_pages=3)
    acc = bench.step_accounting(wl)
    cached = 1000 - 300
    unfused = (-(-cached // 128) * 128) - cached  # 768 - 700 = 68
    assert acc["append_kernel_bytes_fused"] == (unfused + 1) * _row_bytes(wl)
