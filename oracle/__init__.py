"""fp64 CPU oracle for sparse MLA decode (SFA) and the DCP (out, lse) merge.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library under ``deepseek_sparse_mla_sfa_gb300`` never imports it and shares no
code with it.

The arithmetic lives in ``sfa_oracle.c`` (plain C, fp64); this module builds it
with gcc and marshals numpy arrays into it.  The definitions it follows are
stated, with their sources, at the top of ``sfa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsfa_oracle.so")

_lock = threading.Lock()
_lib = None

D_QK = 576  # kv_lora_rank + qk_rope_head_dim
D_V = 512   # kv_lora_rank


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libsfa_oracle.so`` (gcc, -O2, no -ffast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    common = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, ctypes.c_double]
    lib.sfa_oracle_decode.argtypes = common + [P, P, I]
    lib.sfa_oracle_decode.restype = I
    lib.sfa_oracle_decode_splits.argtypes = common + [I, P, P, I]
    lib.sfa_oracle_decode_splits.restype = I
    lib.sfa_oracle_decode_ex.argtypes = common + [I, I, I, P, P, I]
    lib.sfa_oracle_decode_ex.restype = I
    lib.sfa_oracle_decode_sampled.argtypes = common + [I, ctypes.c_long, P, P, P, P, P, I]
    lib.sfa_oracle_decode_sampled.restype = I
    lib.sfa_oracle_decode_sampled_ex.argtypes = common + [I, I, I, ctypes.c_long, P, P, P, P, P, I]
    lib.sfa_oracle_decode_sampled_ex.restype = I
    lib.sfa_oracle_merge.argtypes = [P, P, I, ctypes.c_long, I, P, P]
    lib.sfa_oracle_merge.restype = I
    lib.sfa_oracle_kv_write.argtypes = [P, ctypes.c_long, P, P, ctypes.c_long, I]
    lib.sfa_oracle_kv_write.restype = I
    lib.sfa_oracle_topk.argtypes = [P, ctypes.c_long, P, I, I, I, I, P, I]
    lib.sfa_oracle_topk.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def _as_bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor, or a uint16 numpy array of bf16 bit patterns."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch  # plumbing only: reinterpret bf16 storage as raw bits
    if x.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _as_i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


class Problem:
    """Host copies of one decode problem, in the layouts of the C-ABI.

    q [B*Q, h, 576] bf16, kv [num_blocks, block_size, 576] bf16,
    block_table [B, max_blocks] int32, seq_lens [B] int32, topk_idx [B*Q, top_k] int32.
    """

    def __init__(self, q, kv, block_table, seq_lens, topk_idx, Q: int, scale: float):
        self.q = _as_bf16_bits(q)
        self.kv = _as_bf16_bits(kv)
        self.block_table = _as_i32(block_table)
        self.seq_lens = _as_i32(seq_lens)
        self.topk_idx = _as_i32(topk_idx)
        self.Q = int(Q)
        self.scale = float(scale)
        if self.q.ndim != 3 or self.q.shape[2] != D_QK:
            raise ValueError("q must be [T, h, 576]")
        if self.kv.ndim != 3 or self.kv.shape[2] != D_QK:
            raise ValueError("kv must be [num_blocks, block_size, 576]")
        self.T, self.h = int(self.q.shape[0]), int(self.q.shape[1])
        self.B = int(self.seq_lens.shape[0])
        if self.T != self.B * self.Q:
            raise ValueError("q's first dimension must be B*Q")
        self.num_blocks, self.block_size = int(self.kv.shape[0]), int(self.kv.shape[1])
        self.max_blocks = int(self.block_table.shape[1]) if self.block_table.ndim == 2 else 0
        self.top_k = int(self.topk_idx.shape[1])
        if self.topk_idx.shape[0] != self.T:
            raise ValueError("topk_idx must be [T, top_k]")

    def _common(self):
        return [_ptr(self.q), _ptr(self.kv), _ptr(self.block_table), _ptr(self.seq_lens),
                _ptr(self.topk_idx), self.B, self.Q, self.h, self.top_k, self.num_blocks,
                self.block_size, self.max_blocks, D_QK, D_V, self.scale]


def decode(prob: Problem, nthreads: int = 0):
    """Unsplit SFA decode: returns (out [T, h, 512], lse [T, h]) in float64."""
    lib = _load()
    out = np.zeros((prob.T, prob.h, D_V), dtype=np.float64)
    lse = np.zeros((prob.T, prob.h), dtype=np.float64)
    rc = lib.sfa_oracle_decode(*prob._common(), _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"sfa_oracle_decode failed ({rc})")
    return out, lse


def decode_splits(prob: Problem, n_splits: int, nthreads: int = 0):
    """Per-shard partials: (out_part [n, T, h, 512], lse_part [n, T, h]) in float64."""
    lib = _load()
    out = np.zeros((n_splits, prob.T, prob.h, D_V), dtype=np.float64)
    lse = np.zeros((n_splits, prob.T, prob.h), dtype=np.float64)
    rc = lib.sfa_oracle_decode_splits(*prob._common(), int(n_splits), _ptr(out), _ptr(lse),
                                      int(nthreads))
    if rc != 0:
        raise RuntimeError(f"sfa_oracle_decode_splits failed ({rc})")
    return out, lse


def decode_sampled(prob: Problem, tokens, heads, shards=None, n_splits: int = 1, nthreads: int = 0,
                   interleave: int = 0, bt_per_token: bool = False):
    """Selected (token, head[, shard]) pairs: (out [n, 512], lse [n]) in float64.  The layout
    options are those of decode_ex."""
    if bt_per_token and prob.block_table.shape[0] != prob.T:
        raise ValueError("a per-token block table has one row per query token")
    lib = _load()
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    hh = np.ascontiguousarray(heads, dtype=np.int32)
    r = None if shards is None else np.ascontiguousarray(shards, dtype=np.int32)
    n = int(t.shape[0])
    out = np.zeros((n, D_V), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.sfa_oracle_decode_sampled_ex(*prob._common(), int(n_splits), int(interleave),
                                          int(bool(bt_per_token)), n, _ptr(t), _ptr(hh), _ptr(r),
                                          _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"sfa_oracle_decode_sampled failed ({rc})")
    return out, lse


def decode_ex(prob: Problem, n_splits: int = 1, interleave: int = 0, bt_per_token: bool = False,
              nthreads: int = 0):
    """Per-shard partials with the layout options: shards dealt `interleave` positions at a
    time (0 = contiguous shards) and a block table with one row per query token.  Returns
    (out_part [n, T, h, 512], lse_part [n, T, h]) in float64; n_splits = 1 is unsplit."""
    if bt_per_token and prob.block_table.shape[0] != prob.T:
        raise ValueError("a per-token block table has one row per query token")
    lib = _load()
    out = np.zeros((n_splits, prob.T, prob.h, D_V), dtype=np.float64)
    lse = np.zeros((n_splits, prob.T, prob.h), dtype=np.float64)
    rc = lib.sfa_oracle_decode_ex(*prob._common(), int(n_splits), int(interleave), int(bool(bt_per_token)),
                                  _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"sfa_oracle_decode_ex failed ({rc})")
    return out, lse


def merge(out_part, lse_part):
    """Online-softmax merge over the leading axis: returns (out, lse) in float64."""
    lib = _load()
    op = np.ascontiguousarray(out_part, dtype=np.float64)
    lp = np.ascontiguousarray(lse_part, dtype=np.float64)
    n = int(op.shape[0])
    dv = int(op.shape[-1])
    rows = int(np.prod(op.shape[1:-1])) if op.ndim > 2 else 1
    if lp.shape[0] != n or int(np.prod(lp.shape[1:])) != rows:
        raise ValueError("lse_part must be [n, *rows]")
    out = np.zeros(op.shape[1:], dtype=np.float64)
    lse = np.zeros(lp.shape[1:], dtype=np.float64)
    rc = lib.sfa_oracle_merge(_ptr(op), _ptr(lp), n, rows, dv, _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"sfa_oracle_merge failed ({rc})")
    return out, lse


def kv_write(kv, slot_mapping, rows):
    """The latent-cache write (slot_mapping scatter): returns a copy of `kv` (bf16 bits or
    tensor [num_blocks, block_size, 576]) with row slot_mapping[t] replaced by rows[t]
    for every t whose slot is >= 0.  Raises on a slot past the cache or a repeated slot."""
    lib = _load()
    kvb = _as_bf16_bits(kv).copy()
    sm = _as_i32(slot_mapping)
    rb = _as_bf16_bits(rows)
    D = kvb.shape[-1]
    num_slots = kvb.size // D
    if rb.ndim != 2 or (rb.shape[0] and rb.shape[1] != D) or sm.shape[0] != rb.shape[0]:
        raise ValueError("rows must be [T, D] with one slot per row")
    rc = lib.sfa_oracle_kv_write(_ptr(kvb), num_slots, _ptr(sm), _ptr(rb), int(sm.shape[0]), int(D))
    if rc != 0:
        raise ValueError("slot past the cache or repeated slot")
    return kvb


def uv_proj(out, w_uv):
    """The W_UV up-projection, fp64: y[t, h, v] = sum_c out[t, h, c] * w_uv[h, c, v].

    out [T, h, 512] (float, e.g. the decode output), w_uv [h, 512, 128] as bf16 bits or a
    bf16 tensor.  A plain contraction ("RFC: Context Parallel Modeling for DeepSeek-Style
    Attention", 3.5: W_UV maps each head's 512-wide latent output to its value space),
    done by numpy's einsum in float64.
    """
    if not isinstance(out, np.ndarray):
        out = out.detach().cpu().double().numpy()
    # bf16 bit patterns widen exactly: they are the top half of a float32
    w = (_as_bf16_bits(w_uv).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.einsum("thc,hcv->thv", np.asarray(out, dtype=np.float64), w)


def topk(scores, k: int, seq_lens=None, Q: int = 1, S: Optional[int] = None, nthreads: int = 0) -> np.ndarray:
    """Indexer top-k selection: for each query token t = b*Q + i, the k positions p < L
    (L = min(S, seq_lens[b] - (Q-1-i)), or S without seq_lens) with the largest scores
    under IEEE totalOrder, equal scores taken lower position first, written in ascending
    position and padded with -1.  scores [T, row_stride] float32 (numpy or torch)."""
    if not isinstance(scores, np.ndarray):
        scores = scores.detach().cpu().numpy()
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    if sc.ndim != 2:
        raise ValueError("scores must be [T, row_stride]")
    T, stride = int(sc.shape[0]), int(sc.shape[1])
    S = stride if S is None else int(S)
    sl = None if seq_lens is None else _as_i32(seq_lens)
    if sl is not None:
        B = int(sl.shape[0])
        if B * Q != T:
            raise ValueError("scores must have B*Q rows")
    else:
        if T % Q:
            raise ValueError("T must be a multiple of Q")
        B = T // Q
    out = np.zeros((T, int(k)), dtype=np.int32)
    bits = sc.view(np.uint32)
    rc = _load().sfa_oracle_topk(_ptr(bits), stride, _ptr(sl), B, int(Q), S, int(k), _ptr(out), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"sfa_oracle_topk failed ({rc})")
    return out
