"""CPU checks of the benchmark's work accounting, which every reported rate and roofline
fraction divides by: recounted here entry by entry from the definition (2*h*(576+512)
FLOPs per valid (token, entry, head); gathered rows of 1152 bytes, q, the index lists and
out + lse in fp32, plus the shard partials written and read back when n_splits > 1)."""
import types

import torch

import bench
from deepseek_sparse_mla_sfa_gb300 import workloads


def _recount(w, seq_lens, topk_idx):
    kv = 0
    for t in range(w.T):
        b, i = divmod(t, w.Q)
        L = int(seq_lens[b]) - (w.Q - 1 - i)
        kv += sum(1 for p in topk_idx[t].tolist() if 0 <= p < L)
    flops = 2 * w.h * (576 + 512) * kv
    res = w.T * w.h * (512 + 1) * 4
    decode = kv * 1152 + w.T * w.h * 576 * 2 + w.T * w.top_k * 4 + (w.n_splits * res)
    merge = (w.n_splits + 1) * res if w.n_splits > 1 else 0
    return kv, flops, decode, merge


def test_accounting_matches_a_recount_on_small_workloads():
    for w in (workloads.CONFIGS["tiny"],
              workloads.Workload("acc_mtp", B=3, Q=2, h=8, S=900, S_min=1, top_k=300, n_splits=1,
                                 index_kind="causal", seed=5),
              workloads.Workload("acc_split", B=2, Q=1, h=4, S=500, top_k=128, n_splits=3,
                                 index_kind="uniform", seed=6)):
        inp = workloads.make(w, device="cpu")
        acc = bench.accounting(inp)
        kv, flops, decode, merge = _recount(w, inp.seq_lens, inp.topk_idx)
        assert acc["k_valid_total"] == kv and acc["flops"] == flops, w.name
        assert acc["decode_bytes"] == decode and acc["merge_bytes"] == merge, w.name
        assert acc["gather_bytes"] == kv * 1152


def test_headline_workload_totals():
    # every one of the 2048 entries valid for each of the 64 tokens: 36.5 GFLOP, 177.8 MB
    w = workloads.CONFIGS["sfa_h128"]
    idx = torch.arange(w.top_k, dtype=torch.int32).repeat(w.T, 1)
    inp = types.SimpleNamespace(w=w, seq_lens=torch.full((w.B,), w.S, dtype=torch.int32), topk_idx=idx)
    acc = bench.accounting(inp)
    assert acc["flops"] == 2 * 128 * 1088 * 2048 * 64
    assert abs(acc["flops"] / 1e9 - 36.51) < 0.01
    assert abs(acc["total_bytes"] / 1e6 - 177.8) < 0.1
    assert acc["merge_bytes"] == 0


def test_committed_decode_traffic_matches_the_current_kernel_sources():
    """The roofline's DRAM traffic comes from a committed ncu capture that names the hash
    of the kernel sources it was taken from; a kernel or header change without a new
    capture would leave the bench reporting no traffic for the headline kernel."""
    assert bench.read_traffic("decode", True, "sfa_h128") is not None, (
        "profiles/dram_traffic.txt has no entry for the current decode kernel sources: "
        "recapture the decode profile")
