"""GPU parity of the indexer top-k selection (C ABI sfa_topk) against the oracle:
bit-exact index lists, since the order (IEEE totalOrder, ties to the lower position)
and the output layout (ascending positions, -1 padded) make the answer unique.

* every element on small and mid-size rows: heavy ties, special values, k above the
  candidate count, k = 1, empty and short causal ranges, row strides above S;
* the three top-2048 workloads at full size (every element: the oracle sorts each row);
* the largest supported row (SFA_TOPK_MAX_S);
* the sampled threshold and its fallback to the sweep: chunks whose thresholds differ,
  rows whose top keys crowd the last chunks, negative thresholds, candidates that
  overflow the cluster's buffer;
* the chain into decode: sfa_topk's lists drive sfa_decode to the oracle's attention.
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of

pytestmark = pytest.mark.gpu


def _check(scores, k, seq_lens=None, Q=1, S=None, what=""):
    got = sfa.topk(scores, k, seq_lens=seq_lens, Q=Q, S=S)
    torch.cuda.synchronize()
    ref = oracle.topk(scores, k, seq_lens=seq_lens, Q=Q, S=S)
    g = got.cpu().numpy()
    bad = np.argwhere(g != ref)
    assert bad.size == 0, f"{what}: {bad.shape[0]} entries differ, first at {bad[0].tolist()}"
    assert sfa.last_device_status() == 0
    return g


# (name, T, S, k, kind, stride extra)
SMALL = [
    ("normal_1row", 1, 5000, 300, "normal", 0),
    ("ties_heavy", 4, 9000, 2048, "ties", 0),
    ("special_values", 3, 7000, 1000, "special", 0),
    ("k_above_S", 3, 1000, 2048, "normal", 0),
    ("k_equals_S", 2, 2048, 2048, "normal", 0),
    ("k_one", 5, 4097, 1, "ties", 0),
    ("S_not_multiple_of_4", 3, 4099, 777, "normal", 0),
    ("stride_above_S", 2, 3000, 500, "normal", 36),
    ("S_zero", 2, 0, 16, "normal", 4),
    ("two_slabs_per_thread", 2, 20000, 2048, "ties", 0),
    ("many_rows", 300, 2000, 64, "normal", 0),
]


@pytest.mark.parametrize("name,T,S,k,kind,extra", SMALL, ids=[c[0] for c in SMALL])
def test_small_rows_every_element(name, T, S, k, kind, extra):
    stride = ((S + 3) // 4) * 4 + extra
    sc = workloads.indexer_scores(T, S, "cuda", seed=sum(map(ord, name)), kind=kind, stride=stride)
    _check(sc, k, S=S, what=name)


def test_causal_ranges_with_mtp_tokens():
    # token i of Q sees [0, seq_lens[b] - (Q-1-i)): short, empty and full-length ranges
    seq_lens = torch.tensor([9000, 2049, 2048, 1, 0, 5000], dtype=torch.int32, device="cuda")
    Q, S = 2, 9000
    sc = workloads.indexer_scores(12, S, "cuda", seed=5, kind="ties")
    g = _check(sc, 2048, seq_lens=seq_lens, Q=Q, S=S, what="causal")
    assert np.all(g[6] == -1) and np.all(g[8] == -1) and np.all(g[9] == -1)   # L = 0
    np.testing.assert_array_equal(g[7][:1], [0])
    # seq_lens past S are clipped to S
    _check(sc, 2048, seq_lens=torch.full((6,), 20000, dtype=torch.int32, device="cuda"), Q=Q, S=S,
           what="clipped")


FULL = ["sfa_h128", "mtp", "long_dcp"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_every_element(name):
    """The top-2048 workloads at their full sizes: scores for every position of each
    sequence's cache, each query token choosing over its causal range."""
    w = workloads.CONFIGS[name]
    seq_lens = workloads.make(w, device="cuda").seq_lens
    S = int(seq_lens.max())
    sc = workloads.indexer_scores(w.T, S, "cuda", seed=w.seed)
    g = _check(sc, w.top_k, seq_lens=seq_lens, Q=w.Q, S=S, what=name)
    assert np.all(np.diff(g[:, :16], axis=1) > 0)


def test_largest_supported_row():
    S = 262144
    sc = workloads.indexer_scores(2, S, "cuda", seed=9, kind="ties")
    _check(sc, 2048, S=S, what="max S")
    with pytest.raises(sfa.SfaError):
        sfa.topk(workloads.indexer_scores(1, S + 4, "cuda", seed=9), 2048)


def test_topk_lists_drive_decode_to_the_oracle():
    """Indexer top-k then sparse attention: the kernel's lists, fed to sfa_decode, give
    the oracle's attention over the oracle's lists."""
    w = workloads.Workload("chain", B=3, Q=2, h=64, S=5000, S_min=300, top_k=512, n_splits=1,
                           index_kind="causal", seed=77)
    inp = workloads.make(w, device="cuda")
    S = int(inp.seq_lens.max())
    sc = workloads.indexer_scores(w.T, S, "cuda", seed=78)
    idx = sfa.topk(sc, w.top_k, seq_lens=inp.seq_lens, Q=w.Q, S=S)
    out, lse = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, idx, w.scale, Q=w.Q)
    torch.cuda.synchronize()
    ref_idx = oracle.topk(sc, w.top_k, seq_lens=inp.seq_lens, Q=w.Q, S=S)
    prob = oracle.Problem(inp.q, inp.kv, inp.block_table, inp.seq_lens, ref_idx, w.Q, w.scale)
    ref_out, ref_lse = oracle.decode(prob)
    compare(out, lse, ref_out, ref_lse, "top-k -> decode")


@pytest.mark.parametrize("kind", ["ties", "all_equal"])
def test_full_chunks_with_heavy_ties(kind):
    """Rows held by one CTA each (enough tokens to fill the GPU).  Five-valued scores: a
    fifth of each row ties at the threshold, resolved by position.  All-equal rows: every
    key is a candidate, the lists overflow, and the sweep's per-warp lists overflow too, so
    it compacts the whole chunk; they take the first k positions."""
    T, S, k = 160, 32768, 2048
    if kind == "ties":
        sc = workloads.indexer_scores(T, S, "cuda", seed=21, kind="ties")
    else:
        sc = torch.full((T, S), 0.25, dtype=torch.float32, device="cuda")
    g = _check(sc, k, S=S, what=kind)
    if kind == "all_equal":
        assert np.array_equal(g, np.tile(np.arange(k, dtype=np.int32), (T, 1)))


def _drifting_normal(T, S, seed, drift):
    """N(0, 1) scores whose mean rises linearly by `drift` along the row."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.randn((T, S), generator=gen, device="cuda")
    if drift:
        x += torch.linspace(0.0, drift, S, device="cuda")
    return x


# (name, T, S, k, drift): the kernel first lists the keys above a threshold estimated from a
# sample of each chunk and falls back to sweeping the chunks when that estimate cannot hold
SAMPLED = [
    # 8 CTAs per row whose chunks differ in mean: their thresholds differ, the largest still holds
    ("drift_mild_8_ctas", 6, 65536, 2048, 0.3),
    # the top keys crowd into the last chunks: fewer than k keys reach the largest threshold
    ("drift_strong_8_ctas", 6, 65536, 2048, 4.0),
    # k above half the row: the threshold key is below that of +0
    ("negative_threshold", 200, 8000, 5000, 0.0),
    ("small_k_long_row", 4, 30000, 64, 0.0),
    # the cluster's candidates exceed one chunk's buffer
    ("candidates_overflow", 8, 32768, 20000, 0.0),
    # rows of one CTA each (enough tokens to fill the GPU) whose estimate fails: the sweep
    # without a cluster
    ("drift_strong_one_cta", 160, 32768, 2048, 4.0),
]


@pytest.mark.parametrize("name,T,S,k,drift", SAMPLED, ids=[c[0] for c in SAMPLED])
def test_sampled_threshold_and_its_fallback(name, T, S, k, drift):
    sc = _drifting_normal(T, S, sum(map(ord, name)), drift)
    _check(sc, k, what=name)
