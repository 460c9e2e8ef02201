"""GPU parity of the latent-cache write (slot_mapping scatter, C ABI ``sfa_kv_write``)
against the oracle: a bit copy, so the comparison is exact."""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of, run_cuda

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(seed, num_blocks=40, bs=64, T=300):
    g = torch.Generator().manual_seed(seed)
    kv = torch.randn((num_blocks, bs, 576), generator=g).to(torch.bfloat16)
    rows = torch.randn((T, 576), generator=g).to(torch.bfloat16)
    slots = torch.randperm(num_blocks * bs, generator=g)[:T].to(torch.int32)
    slots[::7] = -1
    return kv, rows, slots


@pytest.mark.parametrize("T", [1, 33, 300])
def test_kv_write_matches_oracle_bit_for_bit(T):
    kv, rows, slots = _case(50 + T, T=T)
    expect = oracle.kv_write(kv, slots.numpy(), rows)
    kv_d = kv.cuda()
    sfa.kv_write(kv_d, slots.cuda(), rows.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kv_d), expect)
    assert sfa.last_device_status() == 0


def test_kv_write_repeated_slot_holds_parts_of_its_rows_and_bad_slot_is_reported():
    kv, rows, _ = _case(60, T=4)
    num_slots = kv.shape[0] * kv.shape[1]
    slots = torch.tensor([5, 5, 9, num_slots], dtype=torch.int32)
    kv_d = kv.cuda()
    sfa.kv_write(kv_d, slots.cuda(), rows.cuda())
    torch.cuda.synchronize()
    assert sfa.last_device_status() == -6          # the slot past the cache is reported
    got = _bits(kv_d).reshape(-1, 576)
    rb = _bits(rows)
    # two writers of slot 5: every 32-bit word of it (the unit a store cannot tear) comes
    # from one of their rows
    w5, w0, w1 = got[5].reshape(-1, 2), rb[0].reshape(-1, 2), rb[1].reshape(-1, 2)
    assert np.all(np.all(w5 == w0, axis=1) | np.all(w5 == w1, axis=1))
    assert np.array_equal(got[9], rb[2])
    before = _bits(kv).reshape(-1, 576)
    untouched = np.setdiff1d(np.arange(num_slots), [5, 9])
    assert np.array_equal(got[untouched], before[untouched])


def test_decode_after_kv_write_matches_oracle():
    # each sequence's last position gets a new latent row, and every query token attends to it
    w = workloads.Workload("kvw", B=4, Q=1, h=128, S=1000, S_min=300, top_k=300, n_splits=1,
                           index_kind="causal", seed=61)
    inp = workloads.make(w, device="cuda")
    bt = inp.block_table.cpu().numpy()
    sl = inp.seq_lens.cpu().numpy()
    bs = inp.kv.shape[1]
    pos = sl - 1
    slots = torch.tensor([int(bt[b, p // bs]) * bs + int(p % bs) for b, p in enumerate(pos)], dtype=torch.int32)
    rows = torch.randn((w.B, 576), generator=torch.Generator().manual_seed(62)).to(torch.bfloat16)
    idx = inp.topk_idx.clone()
    idx[:, 0] = torch.tensor(pos, dtype=torch.int32, device="cuda")
    inp.topk_idx = idx
    kv_new = oracle.kv_write(inp.kv, slots.numpy(), rows)
    sfa.kv_write(inp.kv, slots.cuda(), rows.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(inp.kv), kv_new)
    ref_out, ref_lse = oracle.decode(problem_of(inp))
    out, lse = run_cuda(inp)
    torch.cuda.synchronize()
    compare(out, lse, ref_out, ref_lse, "decode after kv_write")
