"""GPU parity of the W_UV up-projection (C ABI ``sfa_uv_proj``) against the fp64 oracle.

Bound per element, from the arithmetic: out is rounded to bf16 (relative 2^-9), the
bf16 x bf16 products are exact in fp32, the fp32 sum of 512 of them adds at most a few
2^-12 of sum |products|, and the result is rounded to bf16 (relative 2^-9):
    |y - exact| <= 2^-8 * sum_c |out_c * w_cv| + 2^-8 * |exact|
"""
import numpy as np
import pytest
import torch

import deepseek_sparse_mla_sfa_gb300 as sfa
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,h", [(1, 1), (63, 3), (100, 16), (64, 128), (256, 64)])
def test_uv_proj_within_the_rounding_bound(T, h):
    g = torch.Generator().manual_seed(80 + T + h)
    out = (0.3 * torch.randn((T, h, 512), generator=g)).float()
    w = (torch.randn((h, 512, 128), generator=g) / 512 ** 0.5).to(torch.bfloat16)
    y = sfa.uv_proj(out.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert sfa.last_device_status() == 0
    ref = oracle.uv_proj(out.double().numpy(), w)
    absprod = np.einsum("thc,hcv->thv", np.abs(out.double().numpy()), np.abs(w.double().numpy()))
    err = np.abs(y.double().cpu().numpy() - ref)
    bound = 2.0 ** -8 * absprod + 2.0 ** -8 * np.abs(ref) + 1e-6
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"


def test_uv_proj_bounded_wait_timeout_is_reported_and_context_survives():
    """The stall hook makes the W_UV kernel wait on a barrier that nothing completes: the
    wait runs out under a short cap, the kernel reports SFA_ERR_DEVICE_TIMEOUT, drains its
    own loads, and the next call computes the right result."""
    g = torch.Generator().manual_seed(90)
    out = (0.3 * torch.randn((64, 128, 512), generator=g)).float().cuda()
    w = (torch.randn((128, 512, 128), generator=g) / 512 ** 0.5).to(torch.bfloat16).cuda()
    sfa.last_device_status()
    prev = sfa.set_wait_limit(1000)
    prev_stall = sfa.set_stall_injection(True)
    try:
        sfa.uv_proj(out, w)
        status = sfa.last_device_status()
    finally:
        sfa.set_stall_injection(prev_stall)
        sfa.set_wait_limit(prev)
    assert status == -5
    y = sfa.uv_proj(out, w)
    torch.cuda.synchronize()
    assert sfa.last_device_status() == 0
    ref = oracle.uv_proj(out.double().cpu().numpy(), w.cpu())
    absprod = np.einsum("thc,hcv->thv", np.abs(out.double().cpu().numpy()), np.abs(w.double().cpu().numpy()))
    assert np.all(np.abs(y.double().cpu().numpy() - ref) <= 2.0 ** -8 * absprod + 2.0 ** -8 * np.abs(ref) + 1e-6)
