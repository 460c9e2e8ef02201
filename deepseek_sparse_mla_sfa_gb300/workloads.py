"""Seeded synthetic inputs for sparse MLA decode (SFA).

This module only draws random tensors with the shapes, distributions and index
structure of the workloads; it holds none of the attention arithmetic.  Both
the CUDA path (through the tests and the benchmark) and the fp64 oracle are fed
from it.

Shapes follow the paged MLA latent cache of "RFC: MsModeling 支持 Decode Context
Parallel 仿真" (2.1.4.1, 2.1.4.2): q [B*Q, h, 576] bf16 (576 = 512 latent + 64
rope), kv [num_blocks, block_size, 576] bf16 with one latent row per token,
block_table [B, max_blocks_per_seq] int32, seq_lens [B] int32 and a per-token
list of top_k selected positions [B*Q, top_k] int32 (-1 = padding).  The
top-2048 selection follows "vllm-ascend PR #18870 解读" (4.5).

Recipes (values ~ N(0, 1) cast to bf16, scale = 1/sqrt(192)):
  tiny      B=2,   Q=1, h=4,   S=256,     top_k=64,   unique uniform in [0,S), n_splits=2
  dense     B=32,  Q=1, h=16,  S=8192,    top_k=8192, every position in order,   n_splits=4
  sfa_h128  B=64,  Q=1, h=128, S=32768,   top_k=2048, unique uniform in [0,S) unsorted
  mtp       B=128, Q=2, h=64,  S_b~U[1024,65536], seq_lens=S_b+1, top_k=2048;
            token i of a sequence draws unique positions from [0, S_b+i), -1 padded
  long_dcp  B=32,  Q=1, h=128, S=131072,  top_k=2048: 1024 unique from the last 8192
            positions and 1024 unique from the rest, n_splits=8
Physical blocks are a random permutation assigned to the sequences' block-table
rows; unused block-table entries hold -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

D_QK = 576
D_V = 512
SCALE = 1.0 / math.sqrt(192.0)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Q: int
    h: int
    S: int                 # context length (max for the "mtp" recipe)
    top_k: int
    n_splits: int
    index_kind: str        # "uniform" | "dense" | "causal" | "dcp_long"
    block_size: int = 64
    S_min: int = 0         # "causal": per-sequence S_b ~ U[S_min, S]
    recent: int = 8192     # "dcp_long": size of the recent window
    spare_blocks: int = 0  # physical blocks that no sequence owns
    seed: int = 1234
    scale: float = SCALE

    @property
    def T(self) -> int:
        return self.B * self.Q


CONFIGS = {
    "tiny": Workload("tiny", B=2, Q=1, h=4, S=256, top_k=64, n_splits=2, index_kind="uniform",
                     seed=1234 + 1),
    "dense": Workload("dense", B=32, Q=1, h=16, S=8192, top_k=8192, n_splits=4,
                      index_kind="dense", seed=1234 + 2),
    "sfa_h128": Workload("sfa_h128", B=64, Q=1, h=128, S=32768, top_k=2048, n_splits=1,
                         index_kind="uniform", seed=1234 + 3),
    "mtp": Workload("mtp", B=128, Q=2, h=64, S=65536, S_min=1024, top_k=2048, n_splits=1,
                    index_kind="causal", seed=1234 + 4),
    "long_dcp": Workload("long_dcp", B=32, Q=1, h=128, S=131072, top_k=2048, n_splits=8,
                         index_kind="dcp_long", seed=1234 + 5),
}

# the configuration the headline number is quoted on
HEADLINE = "sfa_h128"


@dataclass
class Inputs:
    w: Workload
    q: torch.Tensor            # [T, h, 576] bf16
    kv: torch.Tensor           # [num_blocks, block_size, 576] bf16
    block_table: torch.Tensor  # [B, max_blocks] int32
    seq_lens: torch.Tensor     # [B] int32
    topk_idx: torch.Tensor     # [T, top_k] int32
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _randn_bf16(shape, gen, device, chunk_elems=1 << 28):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def _unique_in_range(rows: int, lo, hi, count: int, width: int, gen, device):
    """For each row, `count` distinct integers drawn uniformly from [lo_r, hi_r)
    (lo/hi scalars or per-row tensors), in random order.  Rows whose range holds
    fewer than `count` integers get all of them followed by -1."""
    lo_t = torch.as_tensor(lo, device=device).expand(rows).to(torch.int64)
    hi_t = torch.as_tensor(hi, device=device).expand(rows).to(torch.int64)
    keys = torch.rand(rows, width, generator=gen, device=device)
    pos = torch.arange(width, device=device).unsqueeze(0) + lo_t.unsqueeze(1)
    keys = torch.where(pos < hi_t.unsqueeze(1), keys, torch.full_like(keys, 2.0))
    k = min(count, width)
    sel_keys, sel = torch.topk(keys, k, dim=1, largest=False, sorted=True)
    vals = torch.where(sel_keys < 2.0, sel + lo_t.unsqueeze(1), torch.full_like(sel, -1))
    # random order among the chosen (topk of random keys is already a random order)
    if k < count:
        vals = torch.cat([vals, torch.full((rows, count - k), -1, device=device, dtype=vals.dtype)], 1)
    return vals.to(torch.int32)


def make(w, device="cuda", seed: Optional[int] = None) -> Inputs:
    """Draw one seeded problem for workload `w` (a Workload or a CONFIGS name)."""
    if isinstance(w, str):
        w = CONFIGS[w]
    seed = w.seed if seed is None else seed
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    B, Q, h, bs = w.B, w.Q, w.h, w.block_size
    T = B * Q
    # per-sequence cache lengths
    if w.index_kind == "causal":
        S_b = torch.randint(w.S_min, w.S + 1, (B,), generator=gen, device=device)
        seq_lens = (S_b + (Q - 1)).to(torch.int32)
    else:
        S_b = torch.full((B,), w.S, device=device, dtype=torch.int64)
        seq_lens = S_b.to(torch.int32)

    # paged cache: each sequence owns ceil(seq_len / bs) blocks, physical ids permuted
    nblk = (seq_lens.to(torch.int64) + bs - 1) // bs
    nblk_host = nblk.cpu()
    max_blocks = max(1, int(nblk_host.max()))
    total = int(nblk_host.sum()) + w.spare_blocks
    perm = torch.randperm(total, generator=gen, device=device).to(torch.int32)
    block_table = torch.full((B, max_blocks), -1, dtype=torch.int32, device=device)
    off = 0
    for b in range(B):
        n = int(nblk_host[b])
        block_table[b, :n] = perm[off:off + n]
        off += n

    q = _randn_bf16((T, h, D_QK), gen, device)
    kv = _randn_bf16((total, bs, D_QK), gen, device)

    # top-k positions
    if w.index_kind == "uniform":
        topk = _unique_in_range(T, 0, w.S, w.top_k, w.S, gen, device)
    elif w.index_kind == "dense":
        if w.top_k != w.S:
            raise ValueError("dense recipe needs top_k == S")
        topk = torch.arange(w.S, device=device, dtype=torch.int32).unsqueeze(0).repeat(T, 1)
    elif w.index_kind == "causal":
        # token i of sequence b draws from [0, S_b + i)
        i = torch.arange(Q, device=device).repeat(B)
        hi = S_b.repeat_interleave(Q) + i
        topk = _unique_in_range(T, 0, hi, w.top_k, int(hi.max()), gen, device)
    elif w.index_kind == "dcp_long":
        half = w.top_k // 2
        recent = _unique_in_range(T, w.S - w.recent, w.S, half, w.recent, gen, device)
        rest = _unique_in_range(T, 0, w.S - w.recent, w.top_k - half, w.S - w.recent, gen, device)
        topk = torch.cat([recent, rest], dim=1)
        # shuffle the two halves together
        order = torch.rand(T, w.top_k, generator=gen, device=device).argsort(dim=1)
        topk = torch.gather(topk, 1, order)
    else:
        raise ValueError(f"unknown index kind {w.index_kind}")

    return Inputs(w=w, q=q, kv=kv, block_table=block_table, seq_lens=seq_lens,
                  topk_idx=topk.contiguous(), meta={"seed": seed})


def small(name: str, **overrides) -> Workload:
    """A copy of a named workload with some fields replaced (for test-sized cases)."""
    return replace(CONFIGS[name], **overrides)


def per_token_block_table(inp: Inputs, shuffle: bool = True, seed: int = 0) -> torch.Tensor:
    """A block table with one row per query token ([B*Q, max_blocks] int32), the layout a
    speculative-decoding batch flattened to one row per token uses ("RFC: MsModeling 支持
    Decode Context Parallel 仿真", 2.1.4.1).  Row t starts as its sequence's row; with
    `shuffle` the sequence's physical blocks are dealt to its logical blocks in a fresh
    random order per token, so that the tokens of one sequence read different cache rows
    for the same position.  Unused entries stay -1."""
    w = inp.w
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    bt = inp.block_table.cpu()
    nblk = ((inp.seq_lens.cpu().to(torch.int64) + w.block_size - 1) // w.block_size).tolist()
    rows = bt.repeat_interleave(w.Q, dim=0).clone()
    if shuffle:
        for t in range(w.T):
            n = nblk[t // w.Q]
            rows[t, :n] = bt[t // w.Q, :n][torch.randperm(n, generator=gen)]
    return rows.contiguous().to(inp.block_table.device)


def indexer_scores(T: int, S: int, device="cuda", seed: int = 0, kind: str = "normal",
                   stride: Optional[int] = None) -> torch.Tensor:
    """Seeded stand-in for the indexer's scores, fp32 [T, stride] (stride = S rounded up to
    a multiple of 4 unless given; columns past S hold +inf, which no selection may pick).
    kind "normal": N(0, 1); "ties": five values {-1, -0.5, 0, 0.5, 1} (heavy ties);
    "special": N(0, 1) with signed zeros, infinities and NaNs mixed in."""
    device = torch.device(device)
    stride = ((S + 3) // 4) * 4 if stride is None else int(stride)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = torch.full((T, stride), float("inf"), dtype=torch.float32, device=device)
    if kind == "normal":
        out[:, :S] = torch.randn((T, S), generator=gen, device=device)
    elif kind == "ties":
        out[:, :S] = torch.randint(-2, 3, (T, S), generator=gen, device=device).float() * 0.5
    elif kind == "special":
        x = torch.randn((T, S), generator=gen, device=device)
        pick = torch.randint(0, 16, (T, S), generator=gen, device=device)
        # +0, -0, +inf, -inf, +NaN (0x7FC00000) and -NaN (0xFFC00000), each 1/16 of the entries
        specials = torch.tensor([0, -0x80000000, 0x7F800000, -0x800000, 0x7FC00000, -0x400000],
                                dtype=torch.int32, device=device).view(torch.float32)
        x = torch.where(pick < 6, specials[pick.clamp(max=5)], x)
        out[:, :S] = x
    else:
        raise ValueError(f"unknown score kind {kind}")
    return out
