"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every
function include/sfa.h declares, and its host-side argument checks return the
documented codes before touching the GPU."""
import ctypes

import pytest

from deepseek_sparse_mla_sfa_gb300 import _lib, build

P0 = ctypes.c_void_p(0)
FAKE = ctypes.c_void_p(1 << 20)   # a non-null, 256-aligned address; never dereferenced here


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_functions_are_all_exported(lib):
    names = _lib.header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/sfa.h but not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.sfa_status_string(code).decode() == name
    assert lib.sfa_status_string(12345).decode() == "SFA_UNKNOWN_STATUS"


def _decode(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, idx=FAKE, B=2, Q=1, h=4, top_k=8, nb=4, bs=64,
             mb=4, scale=0.07, n=1, out=FAKE, lse=FAKE, op=P0, lp=P0, ws=P0, wsb=0, stream=P0)
    a.update(kw)
    return lib.sfa_decode(a["q"], a["kv"], a["bt"], a["sl"], a["idx"], a["B"], a["Q"], a["h"],
                          a["top_k"], a["nb"], a["bs"], a["mb"], a["scale"], a["n"], a["out"],
                          a["lse"], a["op"], a["lp"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=P0), -1), (dict(kv=P0), -1), (dict(idx=P0), -1), (dict(out=P0), -1),
    (dict(h=0), -1), (dict(h=129), -2), (dict(Q=0), -1), (dict(B=-1), -1), (dict(n=0), -1),
    (dict(n=65), -2), (dict(bs=0), -1), (dict(nb=0), -1), (dict(mb=0), -1),
    (dict(scale=float("nan")), -1), (dict(scale=float("inf")), -1),
    (dict(q=ctypes.c_void_p((1 << 20) + 8)), -1),           # q not 16-byte aligned
    (dict(n=2), -1),                                        # partial buffers missing
    (dict(n=2, op=FAKE, lp=FAKE, out=FAKE, lse=P0), -1),     # out without lse
    (dict(B=0), 0), (dict(B=0, q=P0, kv=P0), 0),             # nothing to do
])
def test_host_argument_checks(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_merge_argument_checks(lib):
    m = lib.sfa_lse_merge
    assert m(FAKE, FAKE, 0, 4, 512, FAKE, FAKE, P0) == -1
    assert m(FAKE, FAKE, 65, 4, 512, FAKE, FAKE, P0) == -2
    assert m(FAKE, FAKE, 2, -1, 512, FAKE, FAKE, P0) == -1
    assert m(FAKE, FAKE, 2, 4, 0, FAKE, FAKE, P0) == -1
    assert m(P0, FAKE, 2, 4, 512, FAKE, FAKE, P0) == -1
    assert m(FAKE, FAKE, 2, 0, 512, P0, P0, P0) == 0       # zero rows: nothing to do


def test_workspace_and_staging_sizes(lib):
    assert lib.sfa_decode_workspace_bytes(0, 1, 4, 8, 1) == 0
    ws = lib.sfa_decode_workspace_bytes(64, 1, 128, 2048, 1)
    assert ws % 256 == 0
    st1 = lib.sfa_decode_host_staging_bytes(64, 1, 128, 2048, 512, 1)
    st8 = lib.sfa_decode_host_staging_bytes(64, 1, 128, 2048, 512, 8)
    need = 64 * 128 * 576 * 2 + 64 * 512 * 4 + 64 * 4 + 64 * 2048 * 4 + 64 * 128 * 513 * 4
    assert st1 >= need and st8 >= st1 + 8 * 64 * 128 * 513 * 4
    # a staging buffer that is too small is refused before any copy
    small = lib.sfa_decode_host(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 1, 4, 8, 4, 64, 4, 0.07, 1, FAKE,
                                FAKE, FAKE, 16, P0)
    assert small == -3


def test_wait_limit_hook_roundtrip(lib):
    old = lib.sfa_set_wait_limit(123)
    assert lib.sfa_set_wait_limit(old) == 123


def test_stall_injection_hook_roundtrip(lib):
    old = lib.sfa_set_stall_injection(5)           # any non-zero value turns it on
    assert lib.sfa_set_stall_injection(old) == 1
    assert lib.sfa_set_stall_injection(0) == old


def test_workspace_only_for_the_balanced_schedule(lib):
    # scratch is used only by the 33-64-head kernel when its (token, shard) units outnumber
    # the SMs: two 64 x 512 fp32 partials and 64 (max, sum) pairs per SM plus a counter per
    # unit, each part rounded up to 256 bytes
    for args in ((64, 1, 128, 2048, 1), (32, 1, 128, 2048, 8), (32, 1, 16, 8192, 4), (8, 1, 64, 2048, 1),
                 (300, 1, 32, 2048, 1), (300, 1, 65, 2048, 1), (300, 1, 64, 0, 1)):
        assert lib.sfa_decode_workspace_bytes(*args) == 0, args
    ws = lib.sfa_decode_workspace_bytes(128, 2, 64, 2048, 1)
    per_sm = 2 * (64 * 512 * 4 + 64 * 8)
    counters = (256 * 4 + 255) // 256 * 256
    assert ws > 0 and ws % 256 == 0 and (ws - counters) % per_sm == 0
    n_sms = (ws - counters) // per_sm
    assert 1 <= n_sms < 256
    # the same for 33 heads and for shards as units
    assert lib.sfa_decode_workspace_bytes(128, 2, 33, 2048, 1) == ws
    assert lib.sfa_decode_workspace_bytes(64, 1, 48, 2048, 4) == ws


def _noalloc(lib, out, lse, **kw):
    a = dict(B=2, Q=1, h=4, top_k=8, nb=4, bs=64, mb=4, scale=0.07, n=2)
    a.update(kw)
    return lib.sfa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["Q"], a["h"], a["top_k"], a["nb"],
                                  a["bs"], a["mb"], a["scale"], a["n"], out, lse, P0)


def test_noalloc_host_checks(lib):
    # no result buffer: refused first, whatever else is wrong or empty
    assert _noalloc(lib, P0, FAKE) == -1
    assert _noalloc(lib, FAKE, P0) == -1
    assert _noalloc(lib, P0, P0, B=0) == -1
    assert _noalloc(lib, FAKE, FAKE, Q=0) == -1
    assert _noalloc(lib, FAKE, FAKE, h=129) == -2
    # partials beyond the fixed array: SFA_ERR_WORKSPACE, nothing launched
    assert _noalloc(lib, FAKE, FAKE, B=144, h=128, n=2) == -3
    assert _noalloc(lib, FAKE, FAKE, B=0, h=128, n=2) == 0   # empty batch within the limit


def test_noalloc_binding_refuses_a_q_that_does_not_match_the_batch():
    import torch

    import deepseek_sparse_mla_sfa_gb300 as sfa
    q = torch.zeros((4, 8, 576), dtype=torch.bfloat16)
    kv = torch.zeros((4, 64, 576), dtype=torch.bfloat16)
    bt = torch.zeros((2, 2), dtype=torch.int32)
    sl = torch.full((2,), 64, dtype=torch.int32)
    idx = torch.zeros((4, 16), dtype=torch.int32)
    with pytest.raises(ValueError, match="B / Q / T"):     # T = 4 tokens are 2 sequences x Q=2
        sfa.decode_noalloc(q, kv, bt, sl, idx, 0.07, n_splits=2, Q=1)
    with pytest.raises(ValueError, match="B / Q / T"):
        sfa.decode_noalloc(q, kv, bt, sl, idx, 0.07, n_splits=2, Q=3)
    with pytest.raises(ValueError, match="576"):
        sfa.decode_noalloc(q[:, :, :512].contiguous(), kv, bt, sl, idx, 0.07, Q=2)
    with pytest.raises(ValueError, match="CUDA"):         # consistent shapes, but on the CPU
        sfa.decode_noalloc(q, kv, bt, sl, idx, 0.07, n_splits=2, Q=2)


def _decode_ex(lib, g, flags, **kw):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, idx=FAKE, B=2, Q=1, h=4, top_k=8, nb=4, bs=64,
             mb=4, scale=0.07, n=2, out=FAKE, lse=FAKE, op=FAKE, lp=FAKE, ws=P0, wsb=0, stream=P0)
    a.update(kw)
    return lib.sfa_decode_ex(a["q"], a["kv"], a["bt"], a["sl"], a["idx"], a["B"], a["Q"], a["h"],
                             a["top_k"], a["nb"], a["bs"], a["mb"], a["scale"], a["n"], g, flags,
                             a["out"], a["lse"], a["op"], a["lp"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("g,flags,kw,code", [
    (-1, 0, {}, -1),                 # negative interleave size
    (0, 2, {}, -1),                  # unknown flag bit
    (0, 1 << 30, {}, -1),
    (16, 1, dict(q=P0), -1),         # the common checks still apply
    (16, 1, dict(n=65), -2),
    (16, 1, dict(B=0), 0),           # nothing to do
])
def test_decode_ex_argument_checks(lib, g, flags, kw, code):
    assert _decode_ex(lib, g, flags, **kw) == code


@pytest.mark.parametrize("args,code", [
    (dict(), 0),                                       # B = 0: nothing to do
    (dict(B=2, stride=6), -1),                         # row stride not a multiple of 4
    (dict(B=2, stride=8, S=12), -1),                   # row stride below S
    (dict(B=2, k=0), -1),
    (dict(B=2, Q=0), -1),
    (dict(B=-1), -1),
    (dict(B=2, S=-1), -1),
    (dict(B=2, S=262148, stride=262148), -2),          # above SFA_TOPK_MAX_S
    (dict(B=2, scores=ctypes.c_void_p((1 << 20) + 4)), -1),   # scores not 16-byte aligned
    (dict(B=2, out=P0), -1),
    (dict(B=2, scores=P0), -1),
])
def test_topk_argument_checks(lib, args, code):
    a = dict(scores=FAKE, stride=64, sl=P0, B=0, Q=1, S=64, k=8, out=FAKE)
    a.update(args)
    assert lib.sfa_topk(a["scores"], a["stride"], a["sl"], a["B"], a["Q"], a["S"], a["k"], a["out"], P0) == code


def test_host_plan_argument_checks(lib):
    plan = ctypes.c_void_p(0)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 2, 1, 4, 8, 4, 64, 4, 0.07, 1, FAKE, FAKE, FAKE, 1 << 30]
    assert lib.sfa_host_plan_create(*args, None) == -1                    # no place for the plan
    bad = list(args)
    bad[5] = -1                                                            # B < 0
    assert lib.sfa_host_plan_create(*bad, ctypes.byref(plan)) == -1 and not plan.value
    assert lib.sfa_host_plan_launch(None, P0) == -1
    lib.sfa_host_plan_destroy(None)                                        # ignored
