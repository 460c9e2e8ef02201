"""Hand-derived fixtures under tests/golden/: the oracle (CPU) and the CUDA path (GPU)
against values fixed by the definitions alone.

The pages print no worked example, so each fixture is built from exactly representable
inputs whose result has a closed form (its derivation is stored beside it):

- two_rows_closed_form.json: softmax(scale * q . K^T) . V over two selected rows, with a
  rope column that adds to the score but is not part of V ("vllm-ascend PR #18870 解读",
  4.5; "RFC: MsModeling 支持 Decode Context Parallel 仿真", 2.1.4.1 and 2.1.4.2).
- merge_two_shards.json: the online-softmax merge of two shard partials (same RFC page,
  1.1 and 2.1.1).
- shards_closed_form.json: the partials of two shards, contiguous and dealt one position
  at a time (same RFC page, 2.1.4.1), and their merge.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle

_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
D_QK, D_V = 576, 512
BLOCK_SIZE = 64

# CUDA path tolerances for these fixtures.  The scores are exact in fp32 (products of
# small dyadic numbers); the softmax weights enter the P.V product as bf16, a relative
# error of at most 2**-9 each, so |out - exact| <= 2 * 2**-9 < 4e-3 for outputs in [0, 1].
# lse is formed in fp32 from an exact max and a sum of two exponentials.
ATOL_OUT_GPU = 4e-3
ATOL_LSE_GPU = 1e-4


def _load(name):
    with open(os.path.join(_GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def _two_rows_inputs(h: int):
    """q [1, h, 576], kv [1, 64, 576], block table, seq_lens, topk_idx of the two-row fixture."""
    g = _load("two_rows_closed_form.json")
    q = np.zeros((1, h, D_QK), np.float32)
    for c, v in g["q_nonzero"].items():
        q[0, :, int(c)] = v
    kv = np.zeros((1, BLOCK_SIZE, D_QK), np.float32)
    for r, row in enumerate(g["rows"]):
        for c, v in row.items():
            kv[0, r, int(c)] = v
    bt = np.zeros((1, 1), np.int32)
    seq = np.array([len(g["rows"])], np.int32)
    idx = np.arange(len(g["rows"]), dtype=np.int32)[None, :]
    return g, q, kv, bt, seq, idx


def test_two_rows_closed_form_derivation():
    """The stored values are the closed forms their derivation states."""
    g = _load("two_rows_closed_form.json")
    e2 = math.exp(2.0)
    assert g["expected_out0"] == pytest.approx(e2 / (1.0 + e2), abs=1e-15)
    assert g["expected_lse"] == pytest.approx(math.log1p(e2), abs=1e-15)


def test_oracle_two_rows_closed_form():
    g, q, kv, bt, seq, idx = _two_rows_inputs(h=3)
    import torch
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    prob = oracle.Problem(to_bf16(q), to_bf16(kv), bt, seq, idx, 1, g["scale"])
    out, lse = oracle.decode(prob)
    expect = np.zeros((1, 3, D_V))
    expect[0, :, 0] = g["expected_out0"]
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.full((1, 3), g["expected_lse"]), rtol=0, atol=1e-14)


def test_oracle_merge_two_shards():
    g = _load("merge_two_shards.json")
    n = len(g["lse_part"])
    out_part = np.zeros((n, 1, D_V))
    for s, c in enumerate(g["out_part_unit_columns"]):
        out_part[s, 0, c] = 1.0
    lse_part = np.array(g["lse_part"], np.float64)[:, None]
    out, lse = oracle.merge(out_part, lse_part)
    expect = np.zeros((1, D_V))
    expect[0, :len(g["expected_out"])] = g["expected_out"]
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-15)
    assert lse[0] == pytest.approx(g["expected_lse"], abs=1e-15)


@pytest.mark.gpu
@pytest.mark.parametrize("h", [1, 16, 128])
def test_cuda_two_rows_closed_form(h):
    """Both decode kernels (the small-head and the tensor-core path) give the closed form."""
    import torch
    import deepseek_sparse_mla_sfa_gb300 as sfa
    g, q, kv, bt, seq, idx = _two_rows_inputs(h)
    dev = torch.device("cuda:0")
    out, lse = sfa.decode(torch.from_numpy(q).to(torch.bfloat16).to(dev),
                          torch.from_numpy(kv).to(torch.bfloat16).to(dev),
                          torch.from_numpy(bt).to(dev), torch.from_numpy(seq).to(dev),
                          torch.from_numpy(idx).to(dev), g["scale"])
    torch.cuda.synchronize()
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    expect = np.zeros((1, h, D_V))
    expect[0, :, 0] = g["expected_out0"]
    assert np.abs(o - expect).max() <= ATOL_OUT_GPU
    assert np.abs(l - g["expected_lse"]).max() <= ATOL_LSE_GPU


@pytest.mark.gpu
def test_cuda_merge_two_shards():
    import torch
    import deepseek_sparse_mla_sfa_gb300 as sfa
    g = _load("merge_two_shards.json")
    n = len(g["lse_part"])
    dev = torch.device("cuda:0")
    out_part = torch.zeros((n, 1, D_V), dtype=torch.float32, device=dev)
    for s, c in enumerate(g["out_part_unit_columns"]):
        out_part[s, 0, c] = 1.0
    lse_part = torch.tensor(g["lse_part"], dtype=torch.float32, device=dev)[:, None]
    out, lse = sfa.lse_merge(out_part, lse_part)
    torch.cuda.synchronize()
    expect = np.zeros((1, D_V))
    expect[0, :len(g["expected_out"])] = g["expected_out"]
    # fp32 arithmetic on values near 1: a few ulps
    assert np.abs(out.double().cpu().numpy() - expect).max() <= 1e-6
    assert abs(float(lse[0]) - g["expected_lse"]) <= 1e-6


def _shard_inputs(h: int):
    g = _load("shards_closed_form.json")
    q = np.zeros((1, h, D_QK), np.float32)
    for c, v in g["q_nonzero"].items():
        q[0, :, int(c)] = v
    kv = np.zeros((1, BLOCK_SIZE, D_QK), np.float32)
    for r, row in enumerate(g["rows"]):
        for c, v in row.items():
            kv[0, r, int(c)] = v
    bt = np.zeros((1, 1), np.int32)
    seq = np.array([len(g["rows"])], np.int32)
    idx = np.array([g["topk_idx"]], np.int32)
    return g, q, kv, bt, seq, idx


def _expected_partials(g, interleave: int, h: int):
    part = g["partials"][str(interleave)]
    n = g["n_splits"]
    out = np.zeros((n, 1, h, D_V))
    lse = np.zeros((n, 1, h))
    for r in range(n):
        out[r, 0, :, :2] = part["out01"][r]
        lse[r, 0, :] = part["lse"][r]
    return out, lse


def test_shards_closed_form_derivation():
    g = _load("shards_closed_form.json")
    e2 = math.exp(2.0)
    w = e2 / (1.0 + e2)
    assert g["partials"]["0"]["out01"] == [[pytest.approx(w, abs=1e-15), 0.0], [0.0, 1.0]]
    assert g["partials"]["1"]["out01"] == [[0.0, 0.5], [pytest.approx(w, abs=1e-15),
                                                         pytest.approx(1.0 - w, abs=1e-15)]]
    assert g["partials"]["0"]["lse"] == [pytest.approx(math.log1p(e2), abs=1e-15),
                                         pytest.approx(math.log(2.0), abs=1e-15)]
    assert g["partials"]["1"]["lse"] == [pytest.approx(math.log(2.0), abs=1e-15),
                                         pytest.approx(math.log1p(e2), abs=1e-15)]
    assert g["merged"]["lse"] == pytest.approx(math.log(3.0 + e2), abs=1e-15)
    assert g["merged"]["out01"] == [pytest.approx(e2 / (3.0 + e2), abs=1e-15),
                                    pytest.approx(2.0 / (3.0 + e2), abs=1e-15)]


@pytest.mark.parametrize("interleave", [0, 1])
def test_oracle_shards_closed_form(interleave):
    import torch
    g, q, kv, bt, seq, idx = _shard_inputs(h=2)
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    prob = oracle.Problem(to_bf16(q), to_bf16(kv), bt, seq, idx, 1, g["scale"])
    op, lp = oracle.decode_ex(prob, n_splits=g["n_splits"], interleave=interleave)
    eo, el = _expected_partials(g, interleave, 2)
    np.testing.assert_allclose(op, eo, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lp, el, rtol=0, atol=1e-14)
    mo, ml = oracle.merge(op, lp)
    expect = np.zeros((1, 2, D_V))
    expect[0, :, :2] = g["merged"]["out01"]
    np.testing.assert_allclose(mo, expect, rtol=0, atol=1e-14)
    np.testing.assert_allclose(ml, np.full((1, 2), g["merged"]["lse"]), rtol=0, atol=1e-14)


@pytest.mark.gpu
@pytest.mark.parametrize("interleave", [0, 1])
@pytest.mark.parametrize("h", [1, 128])
def test_cuda_shards_closed_form(h, interleave):
    """Shard partials of both layouts and their merge, on both decode kernels."""
    import torch
    import deepseek_sparse_mla_sfa_gb300 as sfa
    g, q, kv, bt, seq, idx = _shard_inputs(h)
    dev = torch.device("cuda:0")
    args = (torch.from_numpy(q).to(torch.bfloat16).to(dev), torch.from_numpy(kv).to(torch.bfloat16).to(dev),
            torch.from_numpy(bt).to(dev), torch.from_numpy(seq).to(dev), torch.from_numpy(idx).to(dev),
            g["scale"])
    op, lp = sfa.decode(*args, n_splits=g["n_splits"], merge=False, interleave=interleave)
    mo, ml = sfa.decode(*args, n_splits=g["n_splits"], interleave=interleave)
    torch.cuda.synchronize()
    eo, el = _expected_partials(g, interleave, h)
    assert np.abs(op.double().cpu().numpy() - eo).max() <= ATOL_OUT_GPU
    assert np.abs(lp.double().cpu().numpy() - el).max() <= ATOL_LSE_GPU
    expect = np.zeros((1, h, D_V))
    expect[0, :, :2] = g["merged"]["out01"]
    assert np.abs(mo.double().cpu().numpy() - expect).max() <= ATOL_OUT_GPU
    assert np.abs(ml.double().cpu().numpy() - g["merged"]["lse"]).max() <= ATOL_LSE_GPU
