"""GPU check of sfa_decode_noalloc, the entry point for callers that cannot
allocate device memory (an engine whose cache pool owns all free HBM, a plugin
host that passes only inputs and outputs, a loop that cannot pay cudaMalloc's
device-wide synchronisation).  Its shard partials live in a fixed device array
inside the library instead of caller buffers.

The file name puts it last in collection order, so a run that stops at the
first failure has already run every other test.  It must pass on its own in a
fresh process as well as after the rest of the suite.
"""
import ctypes

import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import _lib, workloads
from tests.gpu_helpers import ATOL_LSE, ATOL_OUT, compare, problem_of, run_cuda

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 72 << 20   # SFA_NOALLOC_SCRATCH_BYTES


def _noalloc(inp, out, lse):
    """Call the entry point through the C ABI with caller-owned out/lse only."""
    w = inp.w
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)
    return lib.sfa_decode_noalloc(p(inp.q), p(inp.kv), p(inp.block_table), p(inp.seq_lens),
                                  p(inp.topk_idx), w.B, w.Q, w.h, w.top_k, inp.kv.shape[0],
                                  inp.kv.shape[1], inp.block_table.shape[1], w.scale, w.n_splits,
                                  p(out), p(lse), stream)


def _scratch_need(T, h, n_splits):
    a = lambda x: (x + 255) // 256 * 256
    return a(n_splits * T * h * 512 * 4) + a(n_splits * T * h * 4) if n_splits > 1 else 0


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    cases = [workloads.CONFIGS["long_dcp"],           # 8 shards: partials fill most of the array
             workloads.Workload("noalloc_mtp", B=8, Q=2, h=64, S=6000, S_min=500, top_k=900,
                                n_splits=3, index_kind="causal", seed=31),
             workloads.Workload("noalloc_one_shard", B=4, Q=1, h=128, S=3000, top_k=700,
                                n_splits=1, index_kind="uniform", seed=33)]   # uses no scratch
    for w in cases:
        inp = workloads.make(w, device="cuda")
        ref_out, ref_lse = run_cuda(inp)                 # the existing entry point (sfa_decode)
        for call in range(2):                            # the second call sees the first's scratch
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            assert _noalloc(inp, out, lse) == 0
            torch.cuda.synchronize()
            compare(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                    f"{w.name} noalloc call {call}", ATOL_OUT, ATOL_LSE)
            assert sfa.last_device_status() == 0


def test_noalloc_matches_the_oracle_on_the_sharded_long_context_workload():
    """Independent of the code it wraps: the merged 8-shard result against the fp64 oracle."""
    w = workloads.CONFIGS["long_dcp"]
    inp = workloads.make(w, device="cuda")
    out = torch.full((w.T, w.h, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((w.T, w.h), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(inp, out, lse) == 0
    torch.cuda.synchronize()
    ro, rl = oracle.decode(problem_of(inp))
    compare(out, lse, ro, rl, "long_dcp noalloc vs oracle")
    assert sfa.last_device_status() == 0


def test_noalloc_scratch_limit_is_exact():
    # 2 shards of 128 heads: 525312 bytes of partials per token, so 143 tokens fit in the
    # array and 144 do not
    assert _scratch_need(143, 128, 2) <= SCRATCH_BYTES < _scratch_need(144, 128, 2)
    for B, expect in ((143, 0), (144, -3)):
        w = workloads.Workload(f"limit_{B}", B=B, Q=1, h=128, S=512, top_k=64, n_splits=2,
                               index_kind="uniform", seed=34)
        inp = workloads.make(w, device="cuda")
        out = torch.zeros((w.T, w.h, 512), dtype=torch.float32, device="cuda")
        lse = torch.zeros((w.T, w.h), dtype=torch.float32, device="cuda")
        assert _noalloc(inp, out, lse) == expect, B
        torch.cuda.synchronize()
        if expect == 0:
            ref_out, ref_lse = run_cuda(inp)
            compare(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                    "just under the scratch limit")
        else:   # SFA_ERR_WORKSPACE: nothing was launched
            assert torch.all(out == 0) and torch.all(lse == 0)
    assert sfa.last_device_status() == 0


def test_noalloc_rejects_missing_result_buffers():
    w = workloads.Workload("null_out", B=2, Q=1, h=8, S=256, top_k=32, n_splits=2,
                           index_kind="uniform", seed=35)
    inp = workloads.make(w, device="cuda")
    lse = torch.zeros((w.T, w.h), dtype=torch.float32, device="cuda")
    assert _noalloc(inp, None, lse) == -1
    assert _noalloc(inp, None, None) == -1


def test_noalloc_python_binding_with_two_query_tokens_per_sequence():
    w = workloads.Workload("noalloc_q2", B=6, Q=2, h=32, S=4000, S_min=300, top_k=600, n_splits=2,
                           index_kind="causal", seed=36)
    inp = workloads.make(w, device="cuda")
    out, lse = sfa.decode_noalloc(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx,
                                  w.scale, n_splits=w.n_splits, Q=w.Q)
    torch.cuda.synchronize()
    ro, rl = oracle.decode(problem_of(inp))
    compare(out, lse, ro, rl, "noalloc binding, Q=2")
    with pytest.raises(ValueError):   # Q that does not match the batch is refused, not truncated
        sfa.decode_noalloc(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                           n_splits=w.n_splits, Q=1)
    assert sfa.last_device_status() == 0
