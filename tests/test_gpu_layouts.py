"""GPU parity of the two layout options of sfa_decode_ex against the fp64 oracle:

* interleaved DCP shards: shard r of n holds the cache positions p with
  (p / g) % n == r ("RFC: MsModeling 支持 Decode Context Parallel 仿真", 2.1.4.1,
  cp_kv_cache_interleave_size), every shard partial compared element by element,
  and the merged result against the unsplit oracle;
* a block table with one row per query token (the same page, 2.1.4.1: the table
  flattened for speculative decoding), alone and together with interleaving.

Both kernel paths (tcgen05 and CUDA-core) run every case.
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of, sample_pairs

pytestmark = pytest.mark.gpu

W = workloads.Workload

# (workload, interleave sizes): block-aligned and unaligned sizes, g = 1, g above the
# shard length, several tiles and a ragged tail
INTERLEAVED = [
    (W("il_h128_dcp", B=2, Q=1, h=128, S=20000, recent=2000, top_k=512, n_splits=8,
       index_kind="dcp_long", seed=31), [1, 64, 100]),
    (W("il_h16_dense", B=2, Q=1, h=16, S=1000, top_k=1000, n_splits=4, index_kind="dense", seed=32),
     [16, 300]),
    (W("il_h100_q3", B=2, Q=3, h=100, S=900, S_min=1, top_k=257, n_splits=2, index_kind="causal",
       seed=33), [1, 7]),
    (W("il_h3_bs16", B=2, Q=1, h=3, S=700, top_k=200, n_splits=3, index_kind="uniform",
       block_size=16, seed=34), [5, 64]),
    (W("il_h128_k3000", B=1, Q=1, h=128, S=8192, top_k=3000, n_splits=2, index_kind="uniform",
       seed=35), [32]),
    # more (token, shard) pairs than CTA pairs: the CTA-pair kernel takes groups of shards
    (W("il_h128_groups", B=20, Q=1, h=128, S=8000, top_k=600, n_splits=8, index_kind="uniform",
       seed=36), [16, 1000]),
    # 33-64 heads: more (token, shard) units than SMs (balanced ranges of tiles, units cut
    # between two CTAs), and few units (clusters of 4 CTAs sharing each unit)
    (W("il_h64_balanced", B=90, Q=2, h=64, S=3000, S_min=300, top_k=256, n_splits=2, index_kind="causal",
       seed=37), [16, 100]),
    (W("il_h40_clusters", B=3, Q=1, h=40, S=2000, top_k=500, n_splits=4, index_kind="uniform",
       seed=38), [1, 64]),
]
CASES = [(w, g) for w, gs in INTERLEAVED for g in gs]


# 0 automatic (small-head kernel for h <= 32, stacked-half kernel for h <= 64, CTA pair
# above), 1 CUDA-core, 2 CTA pair for every h (run only where it differs from the automatic
# choice)
@pytest.fixture(params=[0, 1, 2], ids=["auto", "cudacore", "pair"])
def kernel_path(request):
    prev = sfa.set_kernel_path(request.param)
    yield request.param
    sfa.set_kernel_path(prev)


def _skip_duplicate(path, h):
    if path == 2 and h > 64:
        pytest.skip("the automatic path already runs the CTA-pair kernel for h > 64")


def _run(inp, bt, n, g, per_token, merge):
    return sfa.decode(inp.q, inp.kv, bt, inp.seq_lens, inp.topk_idx, inp.w.scale, n_splits=n,
                      Q=inp.w.Q, merge=merge, interleave=g, block_table_per_token=per_token)


def _problem(inp, bt):
    return oracle.Problem(inp.q, inp.kv, bt, inp.seq_lens, inp.topk_idx, inp.w.Q, inp.w.scale)


@pytest.mark.parametrize("w,g", CASES, ids=[f"{w.name}-g{g}" for w, g in CASES])
def test_interleaved_shards_every_element(w, g, kernel_path):
    _skip_duplicate(kernel_path, w.h)
    inp = workloads.make(w, device="cuda")
    prob = problem_of(inp)
    op, lp = _run(inp, inp.block_table, w.n_splits, g, False, merge=False)
    torch.cuda.synchronize()
    rop, rlp = oracle.decode_ex(prob, w.n_splits, interleave=g)
    compare(op, lp, rop, rlp, f"{w.name} g={g} partials")
    # merged: the same attention as the unsplit oracle
    ref_out, ref_lse = oracle.decode(prob)
    out, lse = _run(inp, inp.block_table, w.n_splits, g, False, merge=True)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, f"{w.name} g={g} merged")
    assert sfa.last_device_status() == 0


PER_TOKEN = [
    W("bt_h64_q2", B=3, Q=2, h=64, S=3000, S_min=100, top_k=700, n_splits=1, index_kind="causal", seed=41),
    W("bt_h128_q3", B=2, Q=3, h=128, S=2500, S_min=1, top_k=600, n_splits=1, index_kind="causal", seed=42),
    W("bt_h5_q4_bs16", B=2, Q=4, h=5, S=500, S_min=1, top_k=130, n_splits=1, index_kind="causal",
      block_size=16, seed=43),
    # more than 2048 valid entries: the tensor-core kernel refills its resolved list
    W("bt_h128_q2_k3000", B=1, Q=2, h=128, S=8192, S_min=4000, top_k=3000, n_splits=1, index_kind="causal",
      seed=44),
    # 33-64 heads with more units than SMs: balanced ranges of tiles
    W("bt_h48_balanced", B=80, Q=2, h=48, S=2500, S_min=200, top_k=200, n_splits=1, index_kind="causal",
      seed=45),
]


@pytest.mark.parametrize("w", PER_TOKEN, ids=[w.name for w in PER_TOKEN])
def test_block_table_per_token_every_element(w, kernel_path):
    _skip_duplicate(kernel_path, w.h)
    inp = workloads.make(w, device="cuda")
    bt = workloads.per_token_block_table(inp, shuffle=True, seed=w.seed)
    prob = _problem(inp, bt)
    out, lse = _run(inp, bt, 1, 0, True, merge=True)
    torch.cuda.synchronize()
    rop, rlp = oracle.decode_ex(prob, 1, bt_per_token=True)
    compare(out, lse, rop[0], rlp[0], f"{w.name} per-token table")
    # with 2 interleaved shards as well: partials and merged result
    op, lp = _run(inp, bt, 2, 16, True, merge=False)
    torch.cuda.synchronize()
    rop2, rlp2 = oracle.decode_ex(prob, 2, interleave=16, bt_per_token=True)
    compare(op, lp, rop2, rlp2, f"{w.name} per-token table, interleaved partials")
    mo, ml = _run(inp, bt, 2, 16, True, merge=True)
    torch.cuda.synchronize()
    compare(mo, ml, rop[0], rlp[0], f"{w.name} per-token table, interleaved merged")
    assert sfa.last_device_status() == 0


def test_replicated_per_token_table_is_bit_identical_to_per_sequence(kernel_path):
    """Every token's row equal to its sequence's row: the same rows are read in the same
    order, so the outputs match the per-sequence table bit for bit."""
    w = PER_TOKEN[1]
    inp = workloads.make(w, device="cuda")
    bt = workloads.per_token_block_table(inp, shuffle=False)
    a_out, a_lse = _run(inp, inp.block_table, 1, 0, False, merge=True)
    b_out, b_lse = _run(inp, bt, 1, 0, True, merge=True)
    torch.cuda.synchronize()
    assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)


def test_interleave_size_one_shard_is_the_unsplit_kernel(kernel_path):
    """n_splits = 1 ignores the interleave size: bit-identical to the plain call."""
    w = INTERLEAVED[0][0]
    inp = workloads.make(w, device="cuda")
    a = _run(inp, inp.block_table, 1, 0, False, merge=True)
    b = _run(inp, inp.block_table, 1, 64, False, merge=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_long_dcp_interleaved_full_size_every_element():
    """The 8-shard long-context workload at full size with 64-position interleaving (one
    launch over all shards plus the merge): every merged output against the unsplit
    oracle, and every shard partial against the oracle's interleaved shards (shard r holds
    the positions with (p / 64) % 8 == r)."""
    w = workloads.CONFIGS["long_dcp"]
    inp = workloads.make(w, device="cuda")
    op, lp = _run(inp, inp.block_table, w.n_splits, 64, False, merge=False)
    out, lse = sfa.lse_merge(op, lp)
    torch.cuda.synchronize()
    assert sfa.last_device_status() == 0
    prob = problem_of(inp)
    ref_out, ref_lse = oracle.decode(prob)
    compare(out, lse, ref_out, ref_lse, "long_dcp interleaved merged")
    rop, rlp = oracle.decode_ex(prob, w.n_splits, interleave=64)
    compare(op, lp, rop, rlp, "long_dcp interleaved shard partials")
