"""Invariants of the CUDA path that hold at any size (every kernel):

* permuting the physical cache blocks, with a block table that follows, reads the same
  rows in the same order: bit-identical output;
* permuting each token's index list and padding it with -1 entries changes only the
  rounding;
* any shard count merged by lse_merge gives the unsplit result up to rounding.

Each result is also checked against the fp64 oracle within the parity tolerances.
"""
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of

pytestmark = pytest.mark.gpu

W = workloads.Workload
CASE_WIDE = W("inv", B=3, Q=2, h=128, S=5000, S_min=300, top_k=700, n_splits=1, index_kind="causal", seed=51)
CASE_NARROW = W("inv_h16", B=3, Q=2, h=16, S=5000, S_min=300, top_k=700, n_splits=1, index_kind="causal", seed=52)
CASE_MID = W("inv_h48", B=3, Q=2, h=48, S=5000, S_min=300, top_k=700, n_splits=1, index_kind="causal", seed=53)


# (kernel path, case): the tcgen05 kernels (automatic: CTA pair at h=128, small-head at
# h=16, stacked halves at h=48; forced CTA pair at h=16) and the CUDA-core kernel
@pytest.fixture(params=[(0, CASE_WIDE), (1, CASE_WIDE), (0, CASE_NARROW), (2, CASE_NARROW), (1, CASE_NARROW),
                        (0, CASE_MID)],
                ids=["pair-h128", "cudacore-h128", "small-h16", "pair-h16", "cudacore-h16", "stack-h48"])
def kernel_path(request):
    global CASE
    path, CASE = request.param
    prev = sfa.set_kernel_path(path)
    yield path
    sfa.set_kernel_path(prev)


def _run(inp, kv=None, bt=None, idx=None, n=1):
    return sfa.decode(inp.q, inp.kv if kv is None else kv, inp.block_table if bt is None else bt,
                      inp.seq_lens, inp.topk_idx if idx is None else idx, inp.w.scale, n_splits=n, Q=inp.w.Q)


def test_block_placement_is_bit_invariant(kernel_path):
    inp = workloads.make(CASE, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    nb = inp.kv.shape[0]
    perm = torch.randperm(nb, generator=g, device="cuda")           # block i moves to perm[i]
    kv2 = torch.empty_like(inp.kv)
    kv2[perm] = inp.kv
    bt = inp.block_table
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].to(torch.int32), bt)
    a = _run(inp)
    b = _run(inp, kv=kv2, bt=bt2)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_list_order_and_padding_change_only_rounding(kernel_path):
    inp = workloads.make(CASE, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(6)
    T, k = inp.topk_idx.shape
    order = torch.rand((T, k + 200), generator=g, device="cuda").argsort(dim=1)
    padded = torch.cat([inp.topk_idx, torch.full((T, 200), -1, dtype=torch.int32, device="cuda")], dim=1)
    idx2 = torch.gather(padded, 1, order).contiguous()
    a = _run(inp)
    b = _run(inp, idx=idx2)
    torch.cuda.synchronize()
    assert float((a[0] - b[0]).abs().max()) <= 5e-3
    assert float((a[1] - b[1]).abs().max()) <= 1e-4
    ref_out, ref_lse = oracle.decode(problem_of(inp))
    compare(b[0], b[1], ref_out, ref_lse, "permuted and padded lists")


@pytest.mark.parametrize("n", [2, 3, 8, 64])
def test_any_shard_count_merges_to_the_unsplit_result(n, kernel_path):
    inp = workloads.make(CASE, device="cuda")
    a = _run(inp)
    b = _run(inp, n=n)
    torch.cuda.synchronize()
    assert float((a[0] - b[0]).abs().max()) <= 5e-3
    assert float((a[1] - b[1]).abs().max()) <= 1e-4
    assert sfa.last_device_status() == 0
