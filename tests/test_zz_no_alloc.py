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
from deepseek_sparse_mla_sfa_gb300 import _lib, workloads
from tests.gpu_helpers import ATOL_LSE, ATOL_OUT, compare, run_cuda

pytestmark = pytest.mark.gpu


def _noalloc(inp, out, lse):
    """Call the entry point through the C ABI with caller-owned out/lse only."""
    w = inp.w
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.sfa_decode_noalloc(p(inp.q), p(inp.kv), p(inp.block_table), p(inp.seq_lens),
                                  p(inp.topk_idx), w.B, w.Q, w.h, w.top_k, inp.kv.shape[0],
                                  inp.kv.shape[1], inp.block_table.shape[1], w.scale, w.n_splits,
                                  p(out), p(lse), stream)


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    cases = [workloads.CONFIGS["long_dcp"],           # 8 shards: partials fill most of the array
             workloads.Workload("noalloc_mtp", B=8, Q=2, h=64, S=6000, S_min=500, top_k=900,
                                n_splits=3, index_kind="causal", seed=31)]
    for w in cases:
        inp = workloads.make(w, device="cuda")
        ref_out, ref_lse = run_cuda(inp)                 # the existing entry point (sfa_decode)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(inp, out, lse) == 0
        torch.cuda.synchronize()
        compare(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                w.name + " noalloc", ATOL_OUT, ATOL_LSE)
        assert sfa.last_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = workloads.Workload("too_big", B=64, Q=1, h=128, S=4096, top_k=64, n_splits=8,
                           index_kind="uniform", seed=32)   # 8*64*128*513*4 B > the array
    inp = workloads.make(w, device="cuda")
    out = torch.zeros((w.T, w.h, 512), dtype=torch.float32, device="cuda")
    lse = torch.zeros((w.T, w.h), dtype=torch.float32, device="cuda")
    assert _noalloc(inp, out, lse) == -3                # SFA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(lse == 0)
