"""The library's calls as a serving engine issues them: several streams at once, and
captured into the caller's own CUDA graph and replayed with refilled inputs.  Each
result is compared with the oracle."""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle
from deepseek_sparse_mla_sfa_gb300 import workloads
from tests.gpu_helpers import compare, problem_of

pytestmark = pytest.mark.gpu

W = workloads.Workload


def test_calls_on_concurrent_streams():
    """decode (sharded, merged), topk, uv_proj and kv_write enqueued on four streams with
    no ordering between them: each result equals the oracle's."""
    wd = W("streams_dec", B=6, Q=1, h=128, S=4000, top_k=700, n_splits=3, index_kind="uniform", seed=31)
    inp = workloads.make(wd, device="cuda")
    sc = workloads.indexer_scores(64, 32768, "cuda", seed=32)
    g = torch.Generator().manual_seed(33)
    uo = (0.3 * torch.randn((64, 128, 512), generator=g)).float().cuda()
    uw = (torch.randn((128, 512, 128), generator=g) / 512 ** 0.5).to(torch.bfloat16).cuda()
    kv_c = torch.randn((20, 64, 576), generator=g).to(torch.bfloat16)
    rows = torch.randn((50, 576), generator=g).to(torch.bfloat16)
    slots = torch.randperm(20 * 64, generator=g)[:50].to(torch.int32)
    kv_d = kv_c.cuda()
    rows_d, slots_d = rows.cuda(), slots.cuda()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    with torch.cuda.stream(streams[0]):
        out, lse = sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, wd.scale,
                              n_splits=wd.n_splits, stream=streams[0])
    with torch.cuda.stream(streams[1]):
        idx = sfa.topk(sc, 2048, stream=streams[1])
    with torch.cuda.stream(streams[2]):
        y = sfa.uv_proj(uo, uw, stream=streams[2])
    with torch.cuda.stream(streams[3]):
        sfa.kv_write(kv_d, slots_d, rows_d, stream=streams[3])
    torch.cuda.synchronize()
    assert sfa.last_device_status() == 0
    ro, rl = oracle.decode(problem_of(inp))
    compare(out, lse, ro, rl, "decode on its own stream")
    assert np.array_equal(idx.cpu().numpy(), oracle.topk(sc, 2048))
    ref = oracle.uv_proj(uo.double().cpu().numpy(), uw.cpu())
    absprod = np.einsum("thc,hcv->thv", np.abs(uo.double().cpu().numpy()), np.abs(uw.double().cpu().numpy()))
    assert np.all(np.abs(y.double().cpu().numpy() - ref) <= 2.0 ** -8 * absprod + 2.0 ** -8 * np.abs(ref) + 1e-6)
    got = kv_d.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle.kv_write(kv_c, slots.numpy(), rows))


def test_calls_captured_in_a_caller_graph_and_replayed():
    """topk -> decode (2 shards, merged) captured once in the caller's CUDA graph over
    static buffers; each replay after refilling the inputs gives the oracle's result for
    those inputs."""
    w = W("graph", B=4, Q=2, h=64, S=5000, S_min=2500, top_k=512, n_splits=2, index_kind="causal", seed=34)
    inp = workloads.make(w, device="cuda")
    S = int(inp.seq_lens.max())
    scores = workloads.indexer_scores(w.T, S, "cuda", seed=35)
    idx = torch.empty((w.T, w.top_k), dtype=torch.int32, device="cuda")
    out = torch.empty((w.T, w.h, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.T, w.h), dtype=torch.float32, device="cuda")
    op = torch.empty((w.n_splits, w.T, w.h, 512), dtype=torch.float32, device="cuda")
    lp = torch.empty((w.n_splits, w.T, w.h), dtype=torch.float32, device="cuda")
    q = inp.q.clone()
    # one eager call first (kernel attributes are set outside the capture)
    sfa.topk(scores, w.top_k, seq_lens=inp.seq_lens, Q=w.Q, S=S, out=idx)
    sfa.decode(q, inp.kv, inp.block_table, inp.seq_lens, idx, w.scale, n_splits=w.n_splits, Q=w.Q,
               out=out, lse=lse, out_part=op, lse_part=lp)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            sfa.topk(scores, w.top_k, seq_lens=inp.seq_lens, Q=w.Q, S=S, out=idx, stream=side)
            sfa.decode(q, inp.kv, inp.block_table, inp.seq_lens, idx, w.scale, n_splits=w.n_splits, Q=w.Q,
                       out=out, lse=lse, out_part=op, lse_part=lp, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(3):
        g = torch.Generator(device="cuda").manual_seed(100 + rep)
        scores.copy_(torch.randn(scores.shape, generator=g, device="cuda"))
        q.copy_((torch.randn(q.shape, generator=g, device="cuda")).to(torch.bfloat16))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert sfa.last_device_status() == 0
        ref_idx = oracle.topk(scores, w.top_k, seq_lens=inp.seq_lens, Q=w.Q, S=S)
        assert np.array_equal(idx.cpu().numpy(), ref_idx), f"replay {rep}: top-k lists differ"
        prob = oracle.Problem(q, inp.kv, inp.block_table, inp.seq_lens, ref_idx, w.Q, w.scale)
        ro, rl = oracle.decode(prob)
        compare(out, lse, ro, rl, f"replay {rep}: decode")
