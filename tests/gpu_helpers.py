"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and
the fp64 oracle on the same seeded inputs and compare them."""
from __future__ import annotations

import numpy as np
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads

# tolerances of the CUDA path against the fp64 oracle (max abs error)
ATOL_OUT = 2e-2
ATOL_LSE = 1e-3


def problem_of(inp: workloads.Inputs) -> oracle.Problem:
    return oracle.Problem(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, inp.w.Q,
                          inp.w.scale)


def run_cuda(inp: workloads.Inputs, n_splits=None, merge=True):
    n = inp.w.n_splits if n_splits is None else n_splits
    return sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, inp.w.scale,
                      n_splits=n, Q=inp.w.Q, merge=merge)


def compare(out, lse, ref_out, ref_lse, what="", atol_out=ATOL_OUT, atol_lse=ATOL_LSE):
    """Element-wise check; empty rows must be exactly (0, -inf).  Returns the errors."""
    o = out.detach().double().cpu().numpy() if isinstance(out, torch.Tensor) else np.asarray(out)
    l = lse.detach().double().cpu().numpy() if isinstance(lse, torch.Tensor) else np.asarray(lse)
    ref_out = np.asarray(ref_out)
    ref_lse = np.asarray(ref_lse)
    assert o.shape == ref_out.shape and l.shape == ref_lse.shape, what
    empty = np.isneginf(ref_lse)
    got_empty = np.isneginf(l)
    assert np.array_equal(got_empty, empty), f"{what}: empty-row pattern differs"
    assert np.all(o[empty] == 0.0), f"{what}: empty rows must be exactly zero"
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert np.all(np.isfinite(l[~empty])), f"{what}: non-finite lse"
    e_out = float(np.abs(o - ref_out).max()) if o.size else 0.0
    e_lse = float(np.abs(l[~empty] - ref_lse[~empty]).max()) if (~empty).any() else 0.0
    assert e_out <= atol_out, f"{what}: max |out - oracle| = {e_out:.3e} > {atol_out}"
    assert e_lse <= atol_lse, f"{what}: max |lse - oracle| = {e_lse:.3e} > {atol_lse}"
    return e_out, e_lse


def sample_pairs(T: int, h: int, n: int, seed: int = 0):
    """(token, head) pairs covering the first/last tokens and heads plus random ones."""
    rng = np.random.default_rng(seed)
    t = [0, T - 1, 0, T - 1] + list(rng.integers(0, T, n))
    hh = [0, h - 1, h - 1, 0] + list(rng.integers(0, h, n))
    return np.array(t, np.int32), np.array(hh, np.int32)
