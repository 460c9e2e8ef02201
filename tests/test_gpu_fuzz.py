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


def _grid_case(seed):
    """Batches with more (token, shard) units than the GPU has CTA pairs."""
    rng = np.random.default_rng(8000 + seed)
    h = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(20, 41))
    Q = int(rng.choice([1, 2]))
    n_splits = int(rng.choice([1, 2, 4, 8]))
    S = int(rng.integers(500, 20001))
    top_k = int(rng.integers(64, 601))
    kind = str(rng.choice(["uniform", "causal"]))
    kw = {"S_min": int(rng.integers(0, S + 1))} if kind == "causal" else {}
    w = workloads.Workload(f"grid{seed}", B=B, Q=Q, h=h, S=S, top_k=top_k, n_splits=n_splits,
                           index_kind=kind, block_size=int(rng.choice([16, 64])), seed=9000 + seed, **kw)
    return w, rng


@pytest.mark.parametrize("seed", range(8))
def test_decode_random_multi_wave_grids(seed):
    w, rng = _grid_case(seed)
    inp = workloads.make(w, device="cuda")
    per_token = bool(rng.integers(0, 2))
    bt = workloads.per_token_block_table(inp, seed=seed) if per_token else inp.block_table
    prob = oracle.Problem(inp.q, inp.kv, bt, inp.seq_lens, inp.topk_idx, w.Q, w.scale)
    out, lse = sfa.decode(inp.q, inp.kv, bt, inp.seq_lens, inp.topk_idx, w.scale, n_splits=w.n_splits,
                          Q=w.Q, block_table_per_token=per_token)
    torch.cuda.synchronize()
    if per_token:
        ref_out, ref_lse = oracle.decode_ex(prob, 1, bt_per_token=True)
        ref_out, ref_lse = ref_out[0], ref_lse[0]
    else:
        ref_out, ref_lse = oracle.decode(prob)
    compare(out, lse, ref_out, ref_lse, f"seed {seed}: {w} per_token={per_token}")
    assert sfa.last_device_status() == 0


@pytest.fixture(params=[1, 2], ids=["cudacore", "pair"])
def forced_path(request):
    prev = sfa.set_kernel_path(request.param)
    yield request.param
    sfa.set_kernel_path(prev)


@pytest.mark.parametrize("seed", range(12))
def test_decode_random_shapes_forced_paths(seed, forced_path):
    """The same random shapes on the CUDA-core kernel and, for h <= 64, on the CTA-pair
    kernel (which the automatic choice gives only to h > 64)."""
    w, g, rng = _decode_case(seed)
    if forced_path == 2 and w.h > 64:
        pytest.skip("the automatic path already runs the CTA-pair kernel for h > 64")
    inp = workloads.make(w, device="cuda")
    inp.topk_idx = _salt_indices(inp, rng)
    ref_out, ref_lse = oracle.decode(problem_of(inp))
    out, lse = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                          n_splits=w.n_splits, Q=w.Q, interleave=g)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, f"seed {seed} path {forced_path}: {w} interleave={g}")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("seed", range(12))
def test_lse_merge_random(seed):
    """Shard counts 1 .. 64, row widths with and without 16-byte vectors, empty shards and
    rows whose every shard is empty."""
    rng = np.random.default_rng(11000 + seed)
    n = int(rng.choice([1, 2, 3, 8, 9, 64]))
    rows = int(rng.integers(1, 700))
    dv = int(rng.choice([512, 512, 128, 511, 3, 1]))
    op = rng.standard_normal((n, rows, dv)).astype(np.float32)
    lp = (3.0 * rng.standard_normal((n, rows))).astype(np.float32)
    lp[rng.random((n, rows)) < 0.2] = -np.inf              # empty shards
    lp[:, rng.random(rows) < 0.05] = -np.inf                # rows with no shard at all
    op[np.isneginf(lp)] = 0.0                               # an empty shard's partial is zero
    out, lse = sfa.lse_merge(torch.from_numpy(op).cuda(), torch.from_numpy(lp).cuda())
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.merge(op, lp)
    compare(out, lse, ref_out, ref_lse, f"seed {seed}: n={n} rows={rows} dv={dv}", atol_out=1e-4,
            atol_lse=1e-4)
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_kv_write_random(seed):
    rng = np.random.default_rng(12000 + seed)
    bs = int(rng.choice([1, 16, 64, 256]))
    num_blocks = int(rng.integers(1, 80))
    num_slots = num_blocks * bs
    T = int(rng.integers(0, min(num_slots, 500) + 1))
    g = torch.Generator().manual_seed(13000 + seed)
    kv = torch.randn((num_blocks, bs, 576), generator=g).to(torch.bfloat16)
    rows = torch.randn((T, 576), generator=g).to(torch.bfloat16)
    slots = torch.from_numpy(rng.permutation(num_slots)[:T].astype(np.int32))
    if T:
        slots[torch.from_numpy(rng.random(T) < 0.1)] = -1
    expect = oracle.kv_write(kv, slots.numpy(), rows)
    kv_d = kv.cuda()
    sfa.kv_write(kv_d, slots.cuda(), rows.cuda())
    torch.cuda.synchronize()
    got = kv_d.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, expect), f"seed {seed}: bs={bs} blocks={num_blocks} T={T}"
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_uv_proj_random(seed):
    """Within the rounding bound of the W_UV tests: out rounded to bf16, fp32 sums, y
    rounded to bf16."""
    rng = np.random.default_rng(14000 + seed)
    T = int(rng.integers(1, 300))
    h = int(rng.integers(1, 129))
    g = torch.Generator().manual_seed(15000 + seed)
    out = (0.3 * torch.randn((T, h, 512), generator=g)).float()
    w = (torch.randn((h, 512, 128), generator=g) / 512 ** 0.5).to(torch.bfloat16)
    y = sfa.uv_proj(out.cuda(), w.cuda())
    torch.cuda.synchronize()
    ref = oracle.uv_proj(out.double().numpy(), w)
    absprod = np.einsum("thc,hcv->thv", np.abs(out.double().numpy()), np.abs(w.double().numpy()))
    err = np.abs(y.double().cpu().numpy() - ref)
    bound = 2.0 ** -8 * absprod + 2.0 ** -8 * np.abs(ref) + 1e-6
    assert np.all(err <= bound), f"seed {seed}: T={T} h={h} max err/bound {np.max(err / bound):.3f}"
    assert sfa.last_device_status() == 0


def _decode_case_b(seed):
    """Any head count, block sizes that are not powers of two, long lists (the CTA-pair
    kernel keeps 2048 resolved entries at a time) and scales of either sign around the
    configurations' 1/sqrt(192)."""
    rng = np.random.default_rng(16000 + seed)
    h = int(rng.integers(1, 129))
    B = int(rng.integers(1, 5))
    Q = int(rng.choice([1, 2]))
    bs = int(rng.choice([2, 3, 5, 48, 100, 128, 1000, 64]))
    kind = str(rng.choice(["uniform", "causal"]))
    S = int(rng.integers(1, 9001))
    top_k = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(2048, 6001))]))
    n_splits = int(rng.choice([1, 2, 4]))
    scale = float(rng.choice([1.0, -1.0, 0.0, 0.5, 2.0])) * workloads.SCALE
    kw = {"S_min": int(rng.integers(0, S + 1))} if kind == "causal" else {}
    w = workloads.Workload(f"fuzzb{seed}", B=B, Q=Q, h=h, S=S, top_k=top_k, n_splits=n_splits,
                           index_kind=kind, block_size=bs, seed=17000 + seed, scale=scale, **kw)
    return w, rng


@pytest.mark.parametrize("seed", range(24))
def test_decode_random_shapes_b(seed):
    w, rng = _decode_case_b(seed)
    inp = workloads.make(w, device="cuda")
    inp.topk_idx = _salt_indices(inp, rng)
    prob = problem_of(inp)
    ref_out, ref_lse = oracle.decode(prob)
    out, lse = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                          n_splits=w.n_splits, Q=w.Q)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, f"seed {seed}: {w}")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_decode_noalloc_and_host_entry_points_random(seed):
    """The no-allocation and host-buffer entry points on random shapes, against the oracle."""
    w, g, rng = _decode_case(100 + seed)
    inp = workloads.make(w, device="cuda")
    ref_out, ref_lse = oracle.decode(problem_of(inp))
    out, lse = sfa.decode_noalloc(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                                  n_splits=w.n_splits, Q=w.Q)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, f"noalloc seed {seed}: {w}")
    pin = lambda t: t.cpu().contiguous().pin_memory()
    out_h = torch.full((w.T, w.h, 512), float("nan"), dtype=torch.float32).pin_memory()
    lse_h = torch.full((w.T, w.h), float("nan"), dtype=torch.float32).pin_memory()
    nbytes = sfa.decode_host_staging_bytes(w.B, w.Q, w.h, w.top_k, inp.max_blocks, w.n_splits)
    staging = torch.empty(max(1, nbytes), dtype=torch.uint8, device="cuda")
    sfa.decode_host(pin(inp.q), inp.kv, pin(inp.block_table), pin(inp.seq_lens), pin(inp.topk_idx),
                    w.scale, w.n_splits, w.Q, out_h, lse_h, staging)
    torch.cuda.synchronize()
    compare(out_h, lse_h, ref_out, ref_lse, f"host seed {seed}: {w}")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("S,T", [(98305, 2), (163841, 1), (196609, 3), (229377, 2), (131073, 40),
                                 (65537, 76), (32769, 77), (40000, 3)])
def test_topk_odd_cluster_sizes(S, T):
    """Rows whose plan is a cluster of 3, 5, 6, 7 or 8 CTAs (or 2 at the grid's edge), with
    k around 1 % and 50 % of the row (a threshold key below that of +0)."""
    for k in (max(1, S // 100), S // 2):
        sc = workloads.indexer_scores(T, S, "cuda", seed=S + T + k)
        got = sfa.topk(sc, k, S=S)
        torch.cuda.synchronize()
        ref = oracle.topk(sc, k, S=S)
        bad = np.argwhere(got.cpu().numpy() != ref)
        assert bad.size == 0, f"S={S} T={T} k={k}: {bad.shape[0]} entries differ, first at {bad[0].tolist()}"
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_decode_rescale_stress(seed):
    """q scaled up (scores spread over tens of log2 units) and each list sorted by its
    score, ascending or descending, so the running max grows on almost every tile (and O is
    rescaled) or never after the first."""
    rng = np.random.default_rng(18000 + seed)
    h = int(rng.choice([4, 16, 32, 64, 128]))
    w = workloads.Workload(f"stress{seed}", B=2, Q=1, h=h, S=6000, top_k=int(rng.integers(500, 3000)),
                           n_splits=int(rng.choice([1, 3])), index_kind="uniform", seed=19000 + seed)
    inp = workloads.make(w, device="cuda")
    inp.q = (inp.q.float() * float(rng.choice([2.0, 4.0]))).to(torch.bfloat16)
    prob = problem_of(inp)
    # order each token's list by the score of its first head
    kv = inp.kv.float().reshape(-1, 576)
    q0 = inp.q.float()[:, 0, :]
    for t in range(w.T):
        idx = inp.topk_idx[t].long()
        valid = idx >= 0
        pos = idx[valid]
        blk = inp.block_table[t // w.Q, pos // w.block_size].long()
        rows = kv[blk * w.block_size + pos % w.block_size]
        sc = rows @ q0[t]
        order = torch.argsort(sc, descending=bool(seed % 2))
        inp.topk_idx[t, :pos.numel()] = pos[order].to(torch.int32)
        inp.topk_idx[t, pos.numel():] = -1
    prob = problem_of(inp)
    ref_out, ref_lse = oracle.decode(prob)
    out, lse = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                          n_splits=w.n_splits, Q=w.Q)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, f"seed {seed}: {w}")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("case", ["all_neg_inf", "all_pos_inf", "all_nan", "mixed_inf",
                                  "short_causal_big_cluster", "one_valid_per_cta"])
def test_topk_degenerate_rows(case):
    T, S, k = 4, 70000, 2048
    Q, seq_lens = 1, None
    sc = workloads.indexer_scores(T, S, "cuda", seed=77)
    if case == "all_neg_inf":
        sc[:, :S] = float("-inf")
    elif case == "all_pos_inf":
        sc[:, :S] = float("inf")
    elif case == "all_nan":
        sc[:, :S] = float("nan")
    elif case == "mixed_inf":
        g = torch.Generator(device="cuda").manual_seed(78)
        pick = torch.randint(0, 3, (T, S), generator=g, device="cuda")
        sc[:, :S] = torch.where(pick == 0, float("-inf"), torch.where(pick == 1, float("inf"), sc[:, :S]))
    elif case == "short_causal_big_cluster":
        # the rows plan clusters of several CTAs; the causal ranges reach only the first chunk
        seq_lens = torch.tensor([3000, 2049, 5000, 100], dtype=torch.int32, device="cuda")
    elif case == "one_valid_per_cta":
        k = 1
        seq_lens = torch.tensor([S, 1, 40000, 35000], dtype=torch.int32, device="cuda")
    got = sfa.topk(sc, k, seq_lens=seq_lens, Q=Q, S=S)
    torch.cuda.synchronize()
    ref = oracle.topk(sc, k, seq_lens=seq_lens, Q=Q, S=S)
    bad = np.argwhere(got.cpu().numpy() != ref)
    assert bad.size == 0, f"{case}: {bad.shape[0]} entries differ, first at {bad[0].tolist()}"
    assert sfa.last_device_status() == 0
