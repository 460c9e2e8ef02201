"""Seeded random-shape sweeps of the GPU path against the oracle, every element.

Each case draws its own problem from a seeded generator, so a failure names the seed
that reproduces it:

* decode: head counts across both tcgen05 kernels and their padding (1 .. 128), block
  sizes 1 .. 256, MTP tokens, uniform / causal / long-context index lists, shard counts
  1 .. 8 with contiguous or interleaved shards, and lists salted with entries that must be
  masked (-1, negative, at or past the causal end) and with repeated entries (each entry
  is one attention term);
* top-k: row lengths around the chunk boundaries, k from 1 to past the row, causal ranges,
  strides above S, and score mixes with heavy ties, signed zeros, infinities and NaNs.
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of

pytestmark = pytest.mark.gpu

HEADS = [1, 2, 5, 8, 16, 17, 31, 32, 33, 64, 100, 127, 128]


def _decode_case(seed):
    rng = np.random.default_rng(1000 + seed)
    h = int(rng.choice(HEADS))
    B = int(rng.integers(1, 7))
    Q = int(rng.choice([1, 1, 2, 3]))
    bs = int(rng.choice([1, 16, 64, 64, 256]))
    kind = str(rng.choice(["uniform", "causal", "dcp_long"]))
    S = int(rng.integers(1, 3001)) if kind != "dcp_long" else int(rng.integers(600, 6001))
    top_k = int(rng.integers(1, 1501))
    n_splits = int(rng.choice([1, 1, 2, 3, 5, 8]))
    kw = {}
    if kind == "causal":
        kw["S_min"] = int(rng.integers(0, S + 1))
    if kind == "dcp_long":
        kw["recent"] = int(rng.integers(1, S))
        top_k = max(2, top_k)
    w = workloads.Workload(f"fuzz{seed}", B=B, Q=Q, h=h, S=S, top_k=top_k, n_splits=n_splits,
                           index_kind=kind, block_size=bs, seed=2000 + seed, **kw)
    interleave = int(rng.choice([0, 0, 1, 16, 64])) if n_splits > 1 else 0
    return w, interleave, rng


def _salt_indices(inp, rng):
    """Replace some entries by ones that must be masked, and repeat some others."""
    idx = inp.topk_idx.clone()
    T, k = idx.shape
    Q = inp.w.Q
    # causal end of token t = b*Q + i: seq_lens[b] - (Q-1-i)
    L = [int(inp.seq_lens[t // Q]) - (Q - 1 - t % Q) for t in range(T)]
    n_bad = int(rng.integers(0, max(1, k // 8) + 1))
    n_dup = int(rng.integers(0, max(1, k // 8) + 1))
    for _ in range(n_bad):
        t, j = int(rng.integers(0, T)), int(rng.integers(0, k))
        bad = int(rng.choice([-1, -7, -2147483647, L[t], L[t] + 5, 2147483647]))
        idx[t, j] = bad
    for _ in range(n_dup):
        t, j, j2 = int(rng.integers(0, T)), int(rng.integers(0, k)), int(rng.integers(0, k))
        idx[t, j2] = idx[t, j]
    return idx.contiguous()


@pytest.mark.parametrize("seed", range(32))
def test_decode_random_shapes(seed):
    w, g, rng = _decode_case(seed)
    inp = workloads.make(w, device="cuda")
    inp.topk_idx = _salt_indices(inp, rng)
    prob = problem_of(inp)
    ref_out, ref_lse = oracle.decode(prob)
    out, lse = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                          n_splits=w.n_splits, Q=w.Q, interleave=g)
    torch.cuda.synchronize()
    what = f"seed {seed}: {w} interleave={g}"
    compare(out, lse, ref_out, ref_lse, what)
    if w.n_splits > 1:
        op, lp = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                            n_splits=w.n_splits, Q=w.Q, interleave=g, merge=False)
        rop, rlp = oracle.decode_ex(prob, w.n_splits, interleave=g)
        compare(op, lp, rop, rlp, what + " partials")
    assert sfa.last_device_status() == 0


def _topk_case(seed):
    rng = np.random.default_rng(5000 + seed)
    # row lengths around one chunk, a cluster's chunks and the largest cluster
    S = int(rng.choice([int(rng.integers(0, 300)), int(rng.integers(300, 5000)),
                        int(rng.integers(5000, 40000)), int(rng.integers(40000, 140000))]))
    T = int(rng.choice([1, 2, 5, 16, 64, 160]))
    if S > 40000:
        T = min(T, 16)
    k = int(rng.choice([1, int(rng.integers(1, 64)), int(rng.integers(64, 3000)), S + int(rng.integers(0, 10))]))
    k = max(1, k)
    kind = str(rng.choice(["normal", "normal", "ties", "special"]))
    extra = int(rng.choice([0, 0, 4, 36]))
    Q = int(rng.choice([1, 1, 2]))
    causal = bool(rng.integers(0, 2)) and T % Q == 0
    return S, T, k, kind, extra, Q, causal, rng


@pytest.mark.parametrize("seed", range(40))
def test_topk_random_shapes(seed):
    S, T, k, kind, extra, Q, causal, rng = _topk_case(seed)
    stride = ((S + 3) // 4) * 4 + extra
    sc = workloads.indexer_scores(T, S, "cuda", seed=6000 + seed, kind=kind, stride=stride)
    seq_lens = None
    if causal:
        B = T // Q
        seq_lens = torch.tensor(rng.integers(0, S + 3, B), dtype=torch.int32, device="cuda")
    got = sfa.topk(sc, k, seq_lens=seq_lens, Q=Q if causal else 1, S=S)
    torch.cuda.synchronize()
    ref = oracle.topk(sc, k, seq_lens=seq_lens, Q=Q if causal else 1, S=S)
    g = got.cpu().numpy()
    bad = np.argwhere(g != ref)
    assert bad.size == 0, (f"seed {seed} (S={S} T={T} k={k} kind={kind} stride={stride} Q={Q} "
                           f"causal={causal}): {bad.shape[0]} entries differ, first at {bad[0].tolist()}")
    assert sfa.last_device_status() == 0
