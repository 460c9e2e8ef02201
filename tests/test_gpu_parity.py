"""GPU parity of sfa_decode / sfa_lse_merge (through the C ABI) against the fp64
oracle on the same seeded inputs.

* small and mid-size cases: every output element, every shard partial;
* the five workloads at full size, in the launch configuration the benchmark
  times: every output element and every shard partial.
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of, run_cuda, sample_pairs

pytestmark = pytest.mark.gpu

W = workloads.Workload

# element-by-element cases: several tiles of the kernels, ragged tails, odd head counts
SMALL = [
    workloads.CONFIGS["tiny"],
    workloads.small("tiny", n_splits=1),
    W("h128_ragged", B=3, Q=1, h=128, S=2048, top_k=333, n_splits=1, index_kind="uniform", seed=7),
    W("h128_k2048", B=2, Q=1, h=128, S=8192, top_k=2048, n_splits=1, index_kind="uniform", seed=8),
    W("h64_mtp", B=3, Q=2, h=64, S=3000, S_min=100, top_k=700, n_splits=1, index_kind="causal", seed=9),
    W("h16_dense_splits", B=2, Q=1, h=16, S=1000, top_k=1000, n_splits=4, index_kind="dense", seed=10),
    W("h128_dcp", B=2, Q=1, h=128, S=20000, recent=2000, top_k=512, n_splits=8,
      index_kind="dcp_long", seed=11),
    W("h1", B=2, Q=1, h=1, S=500, top_k=129, n_splits=1, index_kind="uniform", seed=12),
    W("h3_bs16", B=2, Q=1, h=3, S=700, top_k=200, n_splits=3, index_kind="uniform", block_size=16, seed=13),
    W("h33_bs1", B=1, Q=1, h=33, S=300, top_k=150, n_splits=1, index_kind="uniform", block_size=1, seed=14),
    W("h100_q3", B=2, Q=3, h=100, S=900, S_min=1, top_k=257, n_splits=2, index_kind="causal", seed=15),
    W("h65_spare", B=2, Q=1, h=65, S=640, top_k=640, n_splits=1, index_kind="uniform", spare_blocks=5, seed=16),
    # more valid entries than the tcgen05 kernel keeps resolved at once (2048): list refills
    W("h128_k3000", B=1, Q=1, h=128, S=4096, top_k=3000, n_splits=1, index_kind="uniform", seed=17),
    # the largest shard count: 64 shards of 64 positions, many of them empty
    W("h128_n64", B=2, Q=1, h=128, S=4096, top_k=700, n_splits=64, index_kind="uniform", seed=18),
    # a single selected position per token
    W("h128_k1", B=3, Q=1, h=128, S=1000, top_k=1, n_splits=1, index_kind="uniform", seed=19),
    # a list eight times longer than the resolved segment (seven refills), with a ragged tail
    W("h128_k16000", B=1, Q=1, h=128, S=20000, top_k=16000, n_splits=1, index_kind="uniform", seed=20),
    # a large block: 1024 positions per block-table entry
    W("h64_bs1024", B=2, Q=1, h=64, S=5000, top_k=1500, n_splits=2, index_kind="uniform", block_size=1024,
      seed=22),
    # small-head kernel: clusters of 4 (few units), 2 and 1 CTAs per unit, both padded head
    # counts (16, 32), CTAs of a cluster with no tile, a list longer than it keeps resolved
    W("h32_g4", B=3, Q=1, h=32, S=3000, top_k=700, n_splits=1, index_kind="uniform", seed=40),
    W("h16_g2", B=64, Q=1, h=16, S=8192, top_k=2048, n_splits=1, index_kind="uniform", seed=41),
    W("h17_k3000_refill", B=1, Q=1, h=17, S=4096, top_k=3000, n_splits=1, index_kind="uniform", seed=42),
    W("h8_one_tile", B=2, Q=1, h=8, S=500, top_k=40, n_splits=1, index_kind="uniform", seed=43),
    W("h12_mtp_splits", B=5, Q=2, h=12, S=2500, S_min=30, top_k=400, n_splits=3, index_kind="causal", seed=44),
    W("h2_bs16_g1", B=40, Q=1, h=2, S=900, top_k=300, n_splits=2, index_kind="uniform", block_size=16, seed=45),
    # CTA-pair kernel with more (token, shard) pairs than CTA pairs: a unit takes a group of
    # a token's shards (one group per token; two groups per token, with empty shards)
    W("h128_groups1", B=40, Q=1, h=128, S=4096, top_k=600, n_splits=4, index_kind="uniform", seed=46),
    W("h128_groups2_dcp", B=30, Q=1, h=128, S=20000, recent=2000, top_k=512, n_splits=8,
      index_kind="dcp_long", seed=47),
    W("h64_groups_mtp", B=20, Q=2, h=64, S=6000, S_min=40, top_k=700, n_splits=3, index_kind="causal", seed=48),
    # 33-64 heads with more (token, shard) units than SMs: balanced ranges of tiles, units cut
    # between two CTAs and merged through the workspace; ragged lists, short sequences, and
    # shards (many of them empty) as units
    W("h40_balanced", B=80, Q=2, h=40, S=2000, S_min=20, top_k=300, n_splits=1, index_kind="causal", seed=49),
    W("h64_balanced_shards", B=45, Q=1, h=64, S=3000, top_k=333, n_splits=4, index_kind="uniform", seed=50),
    W("h48_balanced_dcp", B=40, Q=1, h=48, S=12000, recent=1500, top_k=257, n_splits=8,
      index_kind="dcp_long", seed=51),
]

# which kernel decode_launches reports per kernel-path setting (0 automatic, 1 CUDA-core,
# 2 CTA-pair tcgen05): 2 = small-head tcgen05, 3 = stacked-half tcgen05, 1 = CTA-pair
# tcgen05, 0 = CUDA-core
def expected_kernel(path, h):
    return {1: 0, 2: 1}.get(path, 2 if h <= 32 else (3 if h <= 64 else 1))


@pytest.fixture(params=[0, 1, 2], ids=["auto", "cudacore", "pair"])
def kernel_path(request):
    prev = sfa.set_kernel_path(request.param)
    yield request.param
    sfa.set_kernel_path(prev)


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_cases_every_element(w, kernel_path):
    if kernel_path == 2 and w.h > 64:
        pytest.skip("the automatic path already runs the CTA-pair kernel for h > 64")
    assert sfa.decode_launches(w.B, w.Q, w.h, w.top_k, w.block_size, w.n_splits)[1] == expected_kernel(kernel_path, w.h)
    inp = workloads.make(w, device="cuda")
    prob = problem_of(inp)
    ref_out, ref_lse = oracle.decode(prob)
    out, lse = run_cuda(inp)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, w.name)
    if w.n_splits > 1:
        op, lp = run_cuda(inp, merge=False)
        rop, rlp = oracle.decode_splits(prob, w.n_splits)
        compare(op, lp, rop, rlp, w.name + " partials")
        # the merge kernel on the partials alone
        mo, ml = sfa.lse_merge(op, lp)
        compare(mo, ml, ref_out, ref_lse, w.name + " lse_merge")
    assert sfa.last_device_status() == 0


FULL = ["tiny", "dense", "sfa_h128", "mtp", "long_dcp"]
# the headline shape with 16 heads, the small-head kernel's bandwidth-bound case
SFA_H16 = W("sfa_h16", B=64, Q=1, h=16, S=32768, top_k=2048, n_splits=1, index_kind="uniform", seed=1234 + 6)


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name):
    """The five workloads at full size, in the launch configuration the benchmark times
    (the whole batch in one launch, units in the kernel's own order): every (token, head)
    output and lse against the fp64 oracle, and for sharded workloads every shard partial
    and the unsplit result too (merged shards == one unsplit pass)."""
    w = workloads.CONFIGS[name]
    inp = workloads.make(w, device="cuda")
    out, lse = run_cuda(inp)
    torch.cuda.synchronize()
    prob = problem_of(inp)
    ro, rl = oracle.decode(prob)
    compare(out, lse, ro, rl, name + " every element")
    if w.n_splits > 1:
        op, lp = run_cuda(inp, merge=False)
        rop, rlp = oracle.decode_splits(prob, w.n_splits)
        compare(op, lp, rop, rlp, name + " every shard partial")
        uo, ul = run_cuda(inp, n_splits=1)
        compare(uo, ul, ro, rl, name + " unsplit")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("path", [0, 2], ids=["small_head", "pair"])
def test_full_size_small_head_every_element(path):
    """B=64, h=16, top_k=2048 over S=32768 on both tcgen05 kernels, every element."""
    prev = sfa.set_kernel_path(path)
    try:
        inp = workloads.make(SFA_H16, device="cuda")
        assert sfa.decode_launches(64, 1, 16, 2048, 64, 1)[1] == (2 if path == 0 else 1)
        out, lse = run_cuda(inp)
        torch.cuda.synchronize()
        ro, rl = oracle.decode(problem_of(inp))
        compare(out, lse, ro, rl, "sfa_h16 every element")
        assert sfa.last_device_status() == 0
    finally:
        sfa.set_kernel_path(prev)


# ------------------------------------------------------------------------------------------
# edge cases and exact index handling
# ------------------------------------------------------------------------------------------
def _inputs(w, **mods):
    inp = workloads.make(w, device="cuda")
    for k, v in mods.items():
        setattr(inp, k, v)
    return inp


def test_empty_rows_and_zero_top_k():
    w = W("edge", B=3, Q=1, h=8, S=300, top_k=40, n_splits=2, index_kind="uniform", seed=21)
    inp = workloads.make(w, device="cuda")
    inp.topk_idx[1] = -1                       # token 1: nothing selected
    inp.topk_idx[2, :20] = 10 ** 6            # token 2: half out of range
    prob = problem_of(inp)
    ro, rl = oracle.decode(prob)
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "empty rows")
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    # top_k = 0
    inp0 = workloads.make(w, device="cuda")
    inp0.topk_idx = torch.empty((w.T, 0), dtype=torch.int32, device="cuda")
    out0, lse0 = run_cuda(inp0)
    assert torch.all(out0 == 0) and torch.all(torch.isneginf(lse0))


def test_zero_tokens_is_a_no_op():
    w = W("zero", B=0, Q=1, h=8, S=64, top_k=4, n_splits=1, index_kind="uniform", seed=22)
    q = torch.empty((0, 8, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 64, 576), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    sl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    idx = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    out, lse = sfa.decode(q, kv, bt, sl, idx, w.scale)
    assert out.shape == (0, 8, 512) and lse.shape == (0, 8)


def test_short_and_empty_sequences_with_mtp():
    # seq_len 0 and seq_len < Q-1: every entry of those tokens is outside the causal range
    w = W("short", B=3, Q=3, h=4, S=200, S_min=1, top_k=30, n_splits=1, index_kind="causal", seed=23)
    inp = workloads.make(w, device="cuda")
    inp.seq_lens[0] = 0
    inp.seq_lens[1] = 1
    inp.topk_idx[:6] = torch.arange(30, device="cuda", dtype=torch.int32) - 3
    prob = problem_of(inp)
    ro, rl = oracle.decode(prob)
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "short sequences")


def test_unreferenced_rows_poisoned_with_nan():
    # every cache row that no valid entry references is NaN: a stray read poisons the output
    w = W("poison", B=2, Q=1, h=128, S=4096, top_k=600, n_splits=2, index_kind="uniform",
          spare_blocks=4, seed=24)
    inp = workloads.make(w, device="cuda")
    inp.topk_idx[:, ::7] = -1
    inp.topk_idx[:, 1::11] = 5000 + torch.arange(inp.topk_idx[:, 1::11].shape[1], device="cuda",
                                                 dtype=torch.int32)
    ref_out, ref_lse = oracle.decode(problem_of(inp))
    keep = torch.zeros(inp.kv.shape[0] * inp.kv.shape[1], dtype=torch.bool, device="cuda")
    bs = w.block_size
    for b in range(w.B):
        p = inp.topk_idx[b]
        p = p[(p >= 0) & (p < inp.seq_lens[b])].long()
        keep[inp.block_table[b, p // bs].long() * bs + p % bs] = True
    flat = inp.kv.view(-1, 576)
    flat[~keep] = float("nan")
    out, lse = run_cuda(inp)
    compare(out, lse, ref_out, ref_lse, "NaN-poisoned cache")
    op, lp = run_cuda(inp, merge=False)
    assert torch.isfinite(op).all()


def test_one_hot_rows_recover_the_rows_read_exactly():
    # q = 0 and the latent row of position p is one-hot at column p % 512 with distinct
    # residues, so round(out * k_valid) is the exact set of rows the kernel read.
    w = W("onehot", B=2, Q=1, h=128, S=4096, top_k=512, n_splits=1, index_kind="uniform", seed=25)
    inp = workloads.make(w, device="cuda")
    inp.q.zero_()
    bs = w.block_size
    expected = torch.zeros((w.B, 512), device="cuda")
    for b in range(w.B):
        pos = torch.randperm(512, device="cuda")[:300] + 512 * torch.randint(0, 8, (300,), device="cuda")
        inp.topk_idx[b] = -1
        inp.topk_idx[b, :300] = pos.to(torch.int32)
        rows = inp.block_table[b, pos // bs].long() * bs + pos % bs
        flat = inp.kv.view(-1, 576)
        flat[rows] = 0
        flat[rows, pos % 512] = 1
        expected[b, pos % 512] = 1
    out, lse = run_cuda(inp)
    for b in range(w.B):
        for hh in (0, 63, 64, 127):
            got = torch.round(out[b, hh] * 300)
            assert torch.equal(got, expected[b]), f"token {b} head {hh}"
    assert torch.allclose(lse, torch.full_like(lse, float(np.log(300))), atol=1e-5)


def test_duplicate_entries_count_per_entry():
    w = W("dup", B=2, Q=1, h=128, S=1024, top_k=300, n_splits=1, index_kind="uniform", seed=26)
    inp = workloads.make(w, device="cuda")
    inp.topk_idx[:, 150:] = inp.topk_idx[:, :150]
    ro, rl = oracle.decode(problem_of(inp))
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "duplicates")


def test_bad_block_table_entry_is_reported_not_read():
    w = W("badblk", B=2, Q=1, h=16, S=512, top_k=64, n_splits=1, index_kind="uniform", seed=27)
    inp = workloads.make(w, device="cuda")
    sfa.last_device_status()
    inp.block_table[0, :] = inp.kv.shape[0] + 1000     # every block of sequence 0 is invalid
    out, lse = run_cuda(inp)
    assert sfa.last_device_status() == -6
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert sfa.last_device_status() == 0                # the status word was cleared


def test_invalid_arguments_raise():
    w = workloads.CONFIGS["tiny"]
    inp = workloads.make(w, device="cuda")
    with pytest.raises(sfa.SfaError):
        sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, float("nan"))
    with pytest.raises(TypeError):
        sfa.decode(inp.q.float(), inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, 0.1)


def test_host_buffer_entry_point_matches_device_entry_point():
    w = W("host", B=4, Q=2, h=64, S=3000, S_min=200, top_k=500, n_splits=2, index_kind="causal", seed=28)
    inp = workloads.make(w, device="cuda")
    out, lse = run_cuda(inp)
    pin = lambda t: t.cpu().pin_memory()
    out_h = torch.empty((w.T, w.h, 512), dtype=torch.float32).pin_memory()
    lse_h = torch.empty((w.T, w.h), dtype=torch.float32).pin_memory()
    nbytes = sfa.decode_host_staging_bytes(w.B, w.Q, w.h, w.top_k, inp.max_blocks, w.n_splits)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sfa.decode_host(pin(inp.q), inp.kv, pin(inp.block_table), pin(inp.seq_lens), pin(inp.topk_idx),
                    w.scale, w.n_splits, w.Q, out_h, lse_h, staging)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out.cpu()) and torch.equal(lse_h, lse.cpu())


@pytest.mark.parametrize("n_splits", [1, 3])
def test_host_buffer_entry_point_in_sequence_groups(n_splits):
    # out >= 4 MiB: the host entry point splits the batch into groups of sequences on
    # helper streams; the result must be the device entry point's, bit for bit
    w = W("host_groups", B=13, Q=2, h=128, S=4000, S_min=300, top_k=400, n_splits=n_splits,
          index_kind="causal", seed=29 + n_splits)
    inp = workloads.make(w, device="cuda")
    out, lse = run_cuda(inp)
    pin = lambda t: t.cpu().pin_memory()
    out_h = torch.full((w.T, w.h, 512), float("nan"), dtype=torch.float32).pin_memory()
    lse_h = torch.full((w.T, w.h), float("nan"), dtype=torch.float32).pin_memory()
    nbytes = sfa.decode_host_staging_bytes(w.B, w.Q, w.h, w.top_k, inp.max_blocks, w.n_splits)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    torch.cuda.synchronize()   # the inputs exist before the side stream reads them
    for stream in (None, side):
        sfa.decode_host(pin(inp.q), inp.kv, pin(inp.block_table), pin(inp.seq_lens), pin(inp.topk_idx),
                        w.scale, w.n_splits, w.Q, out_h, lse_h, staging, stream=stream)
        (side if stream is not None else torch.cuda.current_stream()).synchronize()
        assert torch.equal(out_h, out.cpu()) and torch.equal(lse_h, lse.cpu())
        out_h.fill_(float("nan"))
        lse_h.fill_(float("nan"))
    assert sfa.last_device_status() == 0


def test_tensor_core_kernel_serves_every_workload():
    for name, w in workloads.CONFIGS.items():
        n, tc = sfa.decode_launches(w.B, w.Q, w.h, w.top_k, w.block_size, w.n_splits, merge=False)
        assert tc and n >= 1, name


def test_bounded_wait_timeout_is_reported_and_context_survives():
    # the stall hook makes the kernel wait on a barrier that nothing completes; with a
    # short wait cap that wait runs out, the kernel reports SFA_ERR_DEVICE_TIMEOUT, drains
    # what it has in flight and returns instead of hanging, and the context stays usable
    w = W("timeout", B=2, Q=1, h=128, S=4096, top_k=512, n_splits=1, index_kind="uniform", seed=29)
    inp = workloads.make(w, device="cuda")
    sfa.last_device_status()
    prev = sfa.set_wait_limit(1000)
    prev_stall = sfa.set_stall_injection(True)
    try:
        run_cuda(inp)
        status = sfa.last_device_status()
    finally:
        sfa.set_stall_injection(prev_stall)
        sfa.set_wait_limit(prev)
    assert status == -5
    ro, rl = oracle.decode(problem_of(inp))
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "after timeout")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("h,B", [(16, 2), (32, 64)])
def test_small_head_kernel_timeout_is_reported_and_context_survives(h, B):
    # the small-head kernel with a stalled wait, alone (B=2: clusters of 4) and with clusters
    # of 2: it reports the timeout, every CTA of a cluster still reaches the cluster
    # barriers, and the next call is exact
    w = W("timeout_small", B=B, Q=1, h=h, S=4096, top_k=512, n_splits=1, index_kind="uniform", seed=31)
    inp = workloads.make(w, device="cuda")
    assert sfa.decode_launches(w.B, w.Q, w.h, w.top_k, w.block_size, w.n_splits)[1] == 2
    sfa.last_device_status()
    prev = sfa.set_wait_limit(1000)
    prev_stall = sfa.set_stall_injection(True)
    try:
        run_cuda(inp)
        status = sfa.last_device_status()
    finally:
        sfa.set_stall_injection(prev_stall)
        sfa.set_wait_limit(prev)
    assert status == -5
    ro, rl = oracle.decode(problem_of(inp))
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "small-head kernel after timeout")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("B,Q", [(2, 1), (40, 1), (100, 2)])
def test_stacked_kernel_timeout_is_reported_and_context_survives(B, Q):
    # the 33-64-head kernel with a stalled wait: clusters of 4 (B=2), clusters of 2 (B=40)
    # and balanced ranges of tiles over the SMs (200 units): it reports the timeout, every
    # warp leaves its loop, and the next call is exact (the cut units' counters cleared)
    w = W("timeout_stack", B=B, Q=Q, h=64, S=4096, S_min=600 if Q > 1 else 0, top_k=512, n_splits=1,
          index_kind="causal" if Q > 1 else "uniform", seed=32)
    inp = workloads.make(w, device="cuda")
    assert sfa.decode_launches(w.B, w.Q, w.h, w.top_k, w.block_size, w.n_splits)[1] == 3
    sfa.last_device_status()
    prev = sfa.set_wait_limit(1000)
    prev_stall = sfa.set_stall_injection(True)
    try:
        run_cuda(inp)
        status = sfa.last_device_status()
    finally:
        sfa.set_stall_injection(prev_stall)
        sfa.set_wait_limit(prev)
    assert status == -5
    ro, rl = oracle.decode(problem_of(inp))
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "stacked kernel after timeout")
    assert sfa.last_device_status() == 0


def test_one_poll_wait_cap_reports_or_completes():
    # a cap of one poll may or may not see each barrier complete in time; either way the
    # kernel must return, and the next call is exact
    w = W("onepoll", B=2, Q=1, h=128, S=4096, top_k=512, n_splits=1, index_kind="uniform", seed=30)
    inp = workloads.make(w, device="cuda")
    sfa.last_device_status()
    prev = sfa.set_wait_limit(1)
    try:
        run_cuda(inp)
        status = sfa.last_device_status()
    finally:
        sfa.set_wait_limit(prev)
    assert status in (-5, 0)
    ro, rl = oracle.decode(problem_of(inp))
    out, lse = run_cuda(inp)
    compare(out, lse, ro, rl, "after one-poll cap")
    assert sfa.last_device_status() == 0


@pytest.mark.parametrize("B,n_splits", [(4, 1), (64, 1), (8, 2)])
def test_host_plan_replays_the_host_step(B, n_splits):
    """The captured host step (CUDA graph) gives what decode_host gives, bit for bit, and
    every launch reads the host inputs as they are then: refilled inputs give the
    refilled problem's result.  B=64 takes the grouped path (4 helper streams)."""
    w = W("plan", B=B, Q=1, h=128, S=4096, top_k=512, n_splits=n_splits, index_kind="uniform", seed=29)
    a = workloads.make(w, device="cuda")
    b = workloads.make(w, device="cuda", seed=30)
    pin = lambda t: t.cpu().contiguous().pin_memory()
    q_h, bt_h, sl_h, idx_h = pin(a.q), pin(a.block_table), pin(a.seq_lens), pin(a.topk_idx)
    out_h = torch.empty((w.T, w.h, 512), dtype=torch.float32).pin_memory()
    lse_h = torch.empty((w.T, w.h), dtype=torch.float32).pin_memory()
    nbytes = sfa.decode_host_staging_bytes(w.B, w.Q, w.h, w.top_k, a.max_blocks, w.n_splits)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    plan = sfa.HostPlan(q_h, a.kv, bt_h, sl_h, idx_h, w.scale, w.n_splits, w.Q, out_h, lse_h, staging)
    plan.launch()
    torch.cuda.synchronize()
    ref_out, ref_lse = run_cuda(a)
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref_out.cpu()) and torch.equal(lse_h, ref_lse.cpu())
    # the next step: new queries and index lists in the same pinned buffers (same cache)
    q_h.copy_(b.q.cpu())
    idx_h.copy_(b.topk_idx.cpu())
    plan.launch()
    torch.cuda.synchronize()
    nxt_out, nxt_lse = sfa.decode(b.q, a.kv, a.block_table, a.seq_lens, b.topk_idx, w.scale, n_splits=w.n_splits)
    torch.cuda.synchronize()
    assert torch.equal(out_h, nxt_out.cpu()) and torch.equal(lse_h, nxt_lse.cpu())
    prob = oracle.Problem(b.q, a.kv, a.block_table, a.seq_lens, b.topk_idx, w.Q, w.scale)
    tt, hh = sample_pairs(w.T, w.h, 8, seed=3)
    r_out, r_lse = oracle.decode_sampled(prob, tt, hh)
    compare(out_h[tt, hh].double().numpy(), lse_h[tt, hh].double().numpy(), r_out, r_lse, "plan, second step")
    plan.close()
    assert sfa.last_device_status() == 0
