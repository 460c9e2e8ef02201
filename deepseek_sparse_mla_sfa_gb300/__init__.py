"""GB300 (sm_103a) sparse MLA decode (SFA) with DCP-style split partials.

A thin Python binding over the C ABI of libsfa.so (include/sfa.h).  It only
checks and marshals arguments; every step of the computation runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.

    out, lse = decode(q, kv, block_table, seq_lens, topk_idx, scale)
    out_part, lse_part = decode(..., n_splits=8, merge=False)
    out, lse = lse_merge(out_part, lse_part)
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import SfaError

D_QK = 576
D_V = 512
MAX_HEADS = 128
MAX_SPLITS = 64
BLOCK_TABLE_PER_TOKEN = 1   # sfa_decode_ex flag: one block-table row per query token

__all__ = ["decode", "lse_merge", "decode_host", "decode_host_staging_bytes",
           "workspace_bytes", "decode_noalloc", "decode_launches", "last_device_status", "set_kernel_path",
           "set_wait_limit", "set_stall_injection", "kv_write", "uv_proj", "topk", "HostPlan",
           "SfaError", "D_QK", "D_V", "BLOCK_TABLE_PER_TOKEN"]


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _check_decode_inputs(q, kv, block_table, seq_lens, topk_idx, Q, block_table_per_token=False):
    """The argument checks of every decode entry point: dtypes, ranks, the 576-column
    rows and T == B*Q for q, the index lists and the block table (shapes first, so a bad
    Q is reported even off the GPU), then one CUDA device for everything.  Returns
    (T, h, B, top_k)."""
    for t, name, dt, nd in ((q, "q", torch.bfloat16, 3), (kv, "kv", torch.bfloat16, 3),
                            (block_table, "block_table", torch.int32, 2), (seq_lens, "seq_lens", torch.int32, 1),
                            (topk_idx, "topk_idx", torch.int32, 2)):
        _need(t, name, dt, None, nd)
    T, h, d = q.shape
    if d != D_QK or kv.shape[2] != D_QK:
        raise ValueError("q and kv rows must have 576 columns")
    if int(Q) != Q or Q < 1:
        raise ValueError("Q must be an integer >= 1")
    Q = int(Q)
    B = seq_lens.shape[0]
    bt_rows = T if block_table_per_token else B
    if T != B * Q or topk_idx.shape[0] != T or block_table.shape[0] != bt_rows:
        raise ValueError("inconsistent B / Q / T")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode runs on a CUDA device only")
    for t, name in ((kv, "kv"), (block_table, "block_table"), (seq_lens, "seq_lens"), (topk_idx, "topk_idx")):
        if t.device != dev:
            raise ValueError(f"{name} must be on {dev}, got {t.device}")
    return T, h, B, topk_idx.shape[1]


def workspace_bytes(B: int, Q: int, h: int, top_k: int, n_splits: int) -> int:
    return int(_lib.load().sfa_decode_workspace_bytes(B, Q, h, top_k, n_splits))


def decode(q, kv, block_table, seq_lens, topk_idx, scale: float, n_splits: int = 1, Q: int = 1,
           merge: bool = True, out=None, lse=None, out_part=None, lse_part=None, workspace=None,
           stream=None, interleave: int = 0, block_table_per_token: bool = False):
    """Sparse MLA decode (C ABI ``sfa_decode_ex``; ``sfa_decode`` when both layout options
    are off).

    q [B*Q, h, 576] bf16, kv [num_blocks, block_size, 576] bf16, block_table [B, max_blocks]
    int32 ([B*Q, max_blocks] with block_table_per_token), seq_lens [B] int32, topk_idx
    [B*Q, top_k] int32 (-1 = padding), all on one CUDA device.  interleave = g > 0 deals the
    cache positions to the n_splits shards g at a time (shard r holds (p // g) % n == r);
    0 keeps contiguous shards.  Returns (out [B*Q, h, 512] fp32, lse [B*Q, h] fp32); with
    n_splits > 1 and merge=False returns the shard partials (out_part [n, B*Q, h, 512],
    lse_part [n, B*Q, h]).
    """
    T, h, B, top_k = _check_decode_inputs(q, kv, block_table, seq_lens, topk_idx, Q, block_table_per_token)
    lib = _lib.load()
    dev = q.device
    if interleave < 0:
        raise ValueError("interleave must be >= 0")
    num_blocks, block_size = kv.shape[0], kv.shape[1]
    max_blocks = block_table.shape[1]
    if n_splits == 1 or merge:
        if out is None:
            out = torch.empty((T, h, D_V), dtype=torch.float32, device=dev)
        if lse is None:
            lse = torch.empty((T, h), dtype=torch.float32, device=dev)
        _need(out, "out", torch.float32, dev)
        _need(lse, "lse", torch.float32, dev)
        if tuple(out.shape) != (T, h, D_V) or tuple(lse.shape) != (T, h):
            raise ValueError(f"out must be [{T}, {h}, {D_V}] and lse [{T}, {h}]")
    if n_splits > 1:
        if out_part is None:
            out_part = torch.empty((n_splits, T, h, D_V), dtype=torch.float32, device=dev)
        if lse_part is None:
            lse_part = torch.empty((n_splits, T, h), dtype=torch.float32, device=dev)
        _need(out_part, "out_part", torch.float32, dev)
        _need(lse_part, "lse_part", torch.float32, dev)
    ws_need = int(lib.sfa_decode_workspace_bytes(B, Q, h, top_k, n_splits))
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    flags = BLOCK_TABLE_PER_TOKEN if block_table_per_token else 0
    code = lib.sfa_decode_ex(_ptr(q), _ptr(kv), _ptr(block_table), _ptr(seq_lens), _ptr(topk_idx),
                             B, Q, h, top_k, num_blocks, block_size, max_blocks, float(scale),
                             n_splits, int(interleave), flags,
                             _ptr(out if (n_splits == 1 or merge) else None),
                             _ptr(lse if (n_splits == 1 or merge) else None),
                             _ptr(out_part if n_splits > 1 else None),
                             _ptr(lse_part if n_splits > 1 else None), _ptr(workspace), ws_bytes,
                             _stream_ptr(stream, dev))
    _lib.check("sfa_decode_ex", code)
    if n_splits > 1 and not merge:
        return out_part, lse_part
    return out, lse


def decode_noalloc(q, kv, block_table, seq_lens, topk_idx, scale: float, n_splits: int = 1,
                   Q: int = 1, out=None, lse=None, stream=None):
    """Decode + shard merge without caller-provided scratch (C ABI ``sfa_decode_noalloc``).

    For callers that cannot allocate device memory for shard partials: they live in a
    fixed device array owned by the library (include/sfa.h, SFA_NOALLOC_SCRATCH_BYTES).
    Pass preallocated `out` [B*Q, h, 512] and `lse` [B*Q, h] fp32 to allocate nothing here.
    Calls that overlap on the GPU share that array and race.
    """
    T, h, B, _ = _check_decode_inputs(q, kv, block_table, seq_lens, topk_idx, Q)
    lib = _lib.load()
    dev = q.device
    if out is None:
        out = torch.empty((T, h, D_V), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((T, h), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    _need(lse, "lse", torch.float32, dev)
    if tuple(out.shape) != (T, h, D_V) or tuple(lse.shape) != (T, h):
        raise ValueError(f"out must be [{T}, {h}, {D_V}] and lse [{T}, {h}]")
    code = lib.sfa_decode_noalloc(_ptr(q), _ptr(kv), _ptr(block_table), _ptr(seq_lens),
                                  _ptr(topk_idx), B, Q, h, topk_idx.shape[1], kv.shape[0],
                                  kv.shape[1], block_table.shape[1], float(scale), n_splits,
                                  _ptr(out), _ptr(lse), _stream_ptr(stream, dev))
    _lib.check("sfa_decode_noalloc", code)
    return out, lse


def lse_merge(out_part, lse_part, out=None, lse=None, stream=None):
    """Online-softmax merge over the leading axis (C ABI ``sfa_lse_merge``).

    out_part [n, *rows, dv] fp32, lse_part [n, *rows] fp32 -> (out [*rows, dv], lse [*rows]).
    """
    lib = _lib.load()
    dev = out_part.device
    _need(out_part, "out_part", torch.float32, dev)
    _need(lse_part, "lse_part", torch.float32, dev)
    n = out_part.shape[0]
    dv = out_part.shape[-1]
    rows = lse_part[0].numel() if n > 0 else 0
    if tuple(lse_part.shape) != tuple(out_part.shape[:-1]):
        raise ValueError("lse_part must be out_part's shape without the last axis")
    if out is None:
        out = torch.empty(out_part.shape[1:], dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(lse_part.shape[1:], dtype=torch.float32, device=dev)
    code = lib.sfa_lse_merge(_ptr(out_part), _ptr(lse_part), n, rows, dv, _ptr(out), _ptr(lse),
                             _stream_ptr(stream, dev))
    _lib.check("sfa_lse_merge", code)
    return out, lse


def decode_host_staging_bytes(B, Q, h, top_k, max_blocks, n_splits) -> int:
    return int(_lib.load().sfa_decode_host_staging_bytes(B, Q, h, top_k, max_blocks, n_splits))


def decode_host(q_host, kv, block_table_host, seq_lens_host, topk_idx_host, scale, n_splits,
                Q, out_host, lse_host, staging, stream=None):
    """One decode step with host-resident per-step inputs/outputs (C ABI ``sfa_decode_host``).

    q/block_table/seq_lens/topk_idx and out/lse are (preferably pinned) CPU tensors, kv and
    staging are on the device.  Enqueues copies + kernels on `stream`; synchronise before
    reading out_host / lse_host.
    """
    lib = _lib.load()
    dev = kv.device
    _need(kv, "kv", torch.bfloat16, dev, 3)
    for t, name, dt in ((q_host, "q_host", torch.bfloat16), (block_table_host, "block_table_host", torch.int32),
                        (seq_lens_host, "seq_lens_host", torch.int32), (topk_idx_host, "topk_idx_host", torch.int32),
                        (out_host, "out_host", torch.float32), (lse_host, "lse_host", torch.float32)):
        _need(t, name, dt, torch.device("cpu"))
    T, h, _ = q_host.shape
    B = seq_lens_host.shape[0]
    top_k = topk_idx_host.shape[1]
    code = lib.sfa_decode_host(_ptr(q_host), _ptr(kv), _ptr(block_table_host), _ptr(seq_lens_host),
                               _ptr(topk_idx_host), B, Q, h, top_k, kv.shape[0], kv.shape[1],
                               block_table_host.shape[1], float(scale), n_splits, _ptr(out_host),
                               _ptr(lse_host), _ptr(staging),
                               staging.numel() * staging.element_size(), _stream_ptr(stream, dev))
    _lib.check("sfa_decode_host", code)
    return out_host, lse_host


class HostPlan:
    """One decode_host step captured once as a CUDA graph (C ABI ``sfa_host_plan_*``), for a
    serving loop that reuses its buffers: ``launch()`` enqueues the whole step (input copies,
    kernels, result copies) with one graph launch.

    Arguments as decode_host; the host tensors must be pinned.  Every launch reads the host
    inputs as they are at that moment and writes out_host / lse_host; refill the inputs in
    place between launches and synchronise before reading the results.  The tensors are kept
    alive by the plan.  ``close()`` (or garbage collection) releases it.
    """

    def __init__(self, q_host, kv, block_table_host, seq_lens_host, topk_idx_host, scale, n_splits, Q,
                 out_host, lse_host, staging):
        lib = _lib.load()
        dev = kv.device
        _need(kv, "kv", torch.bfloat16, dev, 3)
        for t, name, dt in ((q_host, "q_host", torch.bfloat16), (block_table_host, "block_table_host", torch.int32),
                            (seq_lens_host, "seq_lens_host", torch.int32),
                            (topk_idx_host, "topk_idx_host", torch.int32),
                            (out_host, "out_host", torch.float32), (lse_host, "lse_host", torch.float32)):
            _need(t, name, dt, torch.device("cpu"))
            if not t.is_pinned():
                raise ValueError(f"{name} must be pinned host memory")
        self._keep = (q_host, kv, block_table_host, seq_lens_host, topk_idx_host, out_host, lse_host, staging)
        self._dev = dev
        T, h, _ = q_host.shape
        B = seq_lens_host.shape[0]
        top_k = topk_idx_host.shape[1]
        plan = ctypes.c_void_p(0)
        code = lib.sfa_host_plan_create(_ptr(q_host), _ptr(kv), _ptr(block_table_host), _ptr(seq_lens_host),
                                        _ptr(topk_idx_host), B, Q, h, top_k, kv.shape[0], kv.shape[1],
                                        block_table_host.shape[1], float(scale), n_splits, _ptr(out_host),
                                        _ptr(lse_host), _ptr(staging), staging.numel() * staging.element_size(),
                                        ctypes.byref(plan))
        _lib.check("sfa_host_plan_create", code)
        self._plan = plan

    def launch(self, stream=None):
        if not self._plan:
            raise ValueError("the plan is closed")
        _lib.check("sfa_host_plan_launch", _lib.load().sfa_host_plan_launch(self._plan, _stream_ptr(stream, self._dev)))

    def close(self):
        if getattr(self, "_plan", None):
            _lib.load().sfa_host_plan_destroy(self._plan)
            self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def uv_proj(out, w_uv, y=None, stream=None):
    """W_UV up-projection (C ABI ``sfa_uv_proj``): y[t, h, v] = sum_c out[t, h, c] * w_uv[h, c, v].

    out [T, h, 512] fp32 (decode's output), w_uv [h, 512, 128] bf16, y [T, h, 128] bf16
    (allocated when None), all on one CUDA device.  Returns y.
    """
    lib = _lib.load()
    dev = out.device
    if dev.type != "cuda":
        raise ValueError("uv_proj runs on a CUDA device only")
    _need(out, "out", torch.float32, dev, 3)
    _need(w_uv, "w_uv", torch.bfloat16, dev, 3)
    T, h, c = out.shape
    if c != D_V or tuple(w_uv.shape) != (h, D_V, 128):
        raise ValueError("out must be [T, h, 512] and w_uv [h, 512, 128]")
    if y is None:
        y = torch.empty((T, h, 128), dtype=torch.bfloat16, device=dev)
    _need(y, "y", torch.bfloat16, dev, 3)
    code = lib.sfa_uv_proj(_ptr(out), _ptr(w_uv), _ptr(y), T, h, _stream_ptr(stream, dev))
    _lib.check("sfa_uv_proj", code)
    return y


def kv_write(kv, slot_mapping, rows, stream=None):
    """Latent-cache write (C ABI ``sfa_kv_write``): kv viewed as [num_blocks*block_size, 576]
    gets row slot_mapping[t] = rows[t] for every t with slot_mapping[t] >= 0, in place.

    kv [num_blocks, block_size, 576] bf16, slot_mapping [T] int32, rows [T, 576] bf16, all on
    one CUDA device.  A slot named twice ends up holding parts of both rows.  Returns kv.
    """
    lib = _lib.load()
    dev = kv.device
    if dev.type != "cuda":
        raise ValueError("kv_write runs on a CUDA device only")
    _need(kv, "kv", torch.bfloat16, dev, 3)
    _need(slot_mapping, "slot_mapping", torch.int32, dev, 1)
    _need(rows, "rows", torch.bfloat16, dev, 2)
    if kv.shape[2] != D_QK or rows.shape[1] != D_QK or rows.shape[0] != slot_mapping.shape[0]:
        raise ValueError("rows must be [T, 576] with one slot per row")
    num_slots = kv.shape[0] * kv.shape[1]
    code = lib.sfa_kv_write(_ptr(kv), num_slots, _ptr(slot_mapping), _ptr(rows), rows.shape[0],
                            _stream_ptr(stream, dev))
    _lib.check("sfa_kv_write", code)
    return kv


def topk(scores, k: int, seq_lens=None, Q: int = 1, S: Optional[int] = None, out=None, stream=None):
    """Indexer top-k selection (C ABI ``sfa_topk``): for each query token t = b*Q + i, the
    positions of the k largest scores among [0, L), L = min(S, seq_lens[b] - (Q-1-i)) (S
    without seq_lens), equal scores lower position first, in ascending position, -1 padded.

    scores [B*Q, row_stride] fp32 (row_stride >= S, a multiple of 4), seq_lens [B] int32 or
    None, out [B*Q, k] int32 (allocated when None), all on one CUDA device.  Returns out,
    the topk_idx layout decode reads.
    """
    lib = _lib.load()
    dev = scores.device
    if dev.type != "cuda":
        raise ValueError("topk runs on a CUDA device only")
    _need(scores, "scores", torch.float32, dev, 2)
    T, stride = scores.shape
    S = stride if S is None else int(S)
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, dev, 1)
        B = seq_lens.shape[0]
        if B * Q != T:
            raise ValueError("scores must have B*Q rows")
    else:
        if T % Q:
            raise ValueError("the number of score rows must be a multiple of Q")
        B = T // Q
    if out is None:
        out = torch.empty((T, int(k)), dtype=torch.int32, device=dev)
    _need(out, "out", torch.int32, dev, 2)
    if tuple(out.shape) != (T, int(k)):
        raise ValueError("out must be [B*Q, k]")
    code = lib.sfa_topk(_ptr(scores), stride, _ptr(seq_lens), B, int(Q), S, int(k), _ptr(out),
                        _stream_ptr(stream, dev))
    _lib.check("sfa_topk", code)
    return out


def decode_launches(B, Q, h, top_k, block_size, n_splits, merge=True):
    """(kernels one decode call enqueues, which kernel serves it: 2 small-head tcgen05,
    3 stacked-half tcgen05, 1 CTA-pair tcgen05, 0 CUDA-core)."""
    tc = ctypes.c_int(0)
    n = int(_lib.load().sfa_decode_launches(B, Q, h, top_k, block_size, n_splits, int(bool(merge)),
                                            ctypes.byref(tc)))
    if n < 0:
        raise ValueError("invalid decode shape")
    return n, int(tc.value)


def last_device_status(stream=None) -> int:
    """Synchronise the stream, then return and clear the device status word (0 = OK)."""
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    return int(lib.sfa_last_device_status(_stream_ptr(stream, dev)))


def set_kernel_path(path: int) -> int:
    """0 = automatic (small-head tcgen05 kernel for h <= 32, stacked-half tcgen05 kernel
    for h <= 64, CTA-pair tcgen05 kernel above), 1 = CUDA-core kernel only, 2 = CTA-pair
    tcgen05 kernel for every h."""
    prev = int(_lib.load().sfa_set_kernel_path(int(path)))
    if prev < 0:
        raise ValueError("path must be 0, 1 or 2")
    return prev


def set_stall_injection(on: bool) -> bool:
    """Test hook (C ABI ``sfa_set_stall_injection``): kernels with bounded waits launched
    afterwards first wait on a barrier nothing completes, so their wait limit runs out and
    they report SFA_ERR_DEVICE_TIMEOUT.  Returns the previous setting."""
    return bool(_lib.load().sfa_set_stall_injection(1 if on else 0))


def set_wait_limit(iterations: int) -> int:
    """Iteration cap of bounded device waits for later launches (0 = default)."""
    return int(_lib.load().sfa_set_wait_limit(int(iterations)))
