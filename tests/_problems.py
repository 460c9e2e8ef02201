"""Small hand-built decode problems for the oracle pins and the parity tests.

Everything here is plain data construction (numpy, torch for bf16 rounding):
placing cache rows, building block tables and index lists.  No attention
arithmetic lives here.
"""
from __future__ import annotations

import numpy as np
import torch

D_QK = 576
D_V = 512


def bf16_bits(x) -> np.ndarray:
    """float array -> uint16 bf16 bit patterns (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Paged:
    """A paged latent cache built from a dense per-sequence array.

    dense [B, S, 576] (float) is placed into kv [num_blocks, bs, 576] through a
    block table whose physical block ids are a permutation (or identity).
    Rows of the cache that no (sequence, position) owns are filled with `fill`.
    """

    def __init__(self, dense: np.ndarray, seq_lens, block_size: int = 64, perm_seed=None,
                 spare_blocks: int = 0, fill=0.0):
        B, S, D = dense.shape
        assert D == D_QK
        self.B, self.S, self.bs = B, S, block_size
        self.seq_lens = np.asarray(seq_lens, dtype=np.int32)
        nblk = [(int(L) + block_size - 1) // block_size for L in self.seq_lens]
        self.max_blocks = max(1, max(nblk))
        total = sum(nblk) + spare_blocks
        ids = np.arange(total, dtype=np.int32)
        if perm_seed is not None:
            ids = np.random.default_rng(perm_seed).permutation(total).astype(np.int32)
        self.block_table = np.full((B, self.max_blocks), -1, dtype=np.int32)
        kv = np.full((total, block_size, D_QK), fill, dtype=np.float32)
        off = 0
        for b in range(B):
            for j in range(nblk[b]):
                phys = ids[off]
                off += 1
                self.block_table[b, j] = phys
                lo = j * block_size
                hi = min(lo + block_size, S)
                if hi > lo:
                    kv[phys, : hi - lo] = dense[b, lo:hi]
        self.kv = bf16_bits(kv)
        self.num_blocks = total


def rng_normal(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)
