"""Failure detection on the GPU without a GPU fault: with the test hook on, the
kernel's copy warp issues nothing, so every other role's bounded wait runs out
(about one second).  The kernel must record ATTN_ERR_TIMEOUT in the device
status word, free its tensor memory and return; the context stays usable and
the next normal call is correct."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import CAUSAL, DENSE, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def af():
    import attention_forward_15_gb300 as m
    from attention_forward_15_gb300 import _build_ext
    _build_ext.build()
    lib = m.load_library()
    lib.attn_debug_inject.restype = ctypes.c_int
    lib.attn_debug_inject.argtypes = [ctypes.c_int]
    return m


@pytest.mark.parametrize("D,mask,dt", [(64, DENSE, torch.float16), (128, CAUSAL, torch.bfloat16),
                                       (256, DENSE, torch.bfloat16)])
def test_timeout_is_reported_and_recovered(af, D, mask, dt):
    lib = af.load_library()
    dev = torch.device("cuda", 0)
    q, k, v = make_qkv(1, 2, 512, D, dt, seed=5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    assert af.last_device_status(0)[0] == 0
    assert lib.attn_debug_inject(1) == 0
    try:
        af.fwd(qd, kd, vd, mask, 0, 1.0 / math.sqrt(D))
        torch.cuda.synchronize()
    finally:
        assert lib.attn_debug_inject(0) == 0
    st, detail = af.last_device_status(0)
    assert st == 7, f"expected ATTN_ERR_TIMEOUT, got {st} (detail {detail:#x})"
    assert (detail >> 8) & 0xff != 0                     # a wait site was recorded
    assert af.last_device_status(0)[0] == 0              # the query clears the word
    # the context is still usable and the next call is right
    o, lse = af.fwd(qd, kd, vd, mask, 0, 1.0 / math.sqrt(D))
    torch.cuda.synchronize()
    O_ref, l_ref = oracle.attention(q, k, v, mask, 0, 1.0 / math.sqrt(D))
    tol = 4e-3 if dt == torch.float16 else 1.6e-2
    assert np.abs(o.double().cpu().numpy() - O_ref).max() <= tol
    assert np.abs(lse.double().cpu().numpy() - l_ref).max() <= 1e-3
    assert af.last_device_status(0)[0] == 0


@pytest.mark.parametrize("D", [64, 256])
def test_bwd_timeout_is_reported_and_recovered(af, D):
    """The same for the backward's two tile kernels (one small head, so every
    CTA's wait runs out at once; D = 256 runs the half-tile ring): the timeout
    is reported with a wait site, and the next backward on the same context is
    right."""
    lib = af.load_library()
    dev = torch.device("cuda", 0)
    q, k, v = make_qkv(1, 1, 256, D, torch.float16, seed=6)
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(7)).to(q.dtype)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    o, lse = af.fwd(qd, kd, vd, CAUSAL)
    torch.cuda.synchronize()
    assert af.last_device_status(0)[0] == 0
    assert lib.attn_debug_inject(1) == 0
    try:
        af.bwd(qd, kd, vd, o, lse, gd, CAUSAL)
        torch.cuda.synchronize()
    finally:
        assert lib.attn_debug_inject(0) == 0
    st, detail = af.last_device_status(0)
    assert st == 7, f"expected ATTN_ERR_TIMEOUT, got {st} (detail {detail:#x})"
    assert (detail >> 8) & 0xff != 0
    dq, dk, dv = af.bwd(qd, kd, vd, o, lse, gd, CAUSAL)
    torch.cuda.synchronize()
    assert af.last_device_status(0)[0] == 0
    ref = oracle.attention_bwd(q, k, v, g, CAUSAL, 0, float(np.float32(1.0 / math.sqrt(D))), bounds=True)
    u = 2.0 ** -11
    for got, want, bnd in zip((dq, dk, dv), ref[:3], ref[3:]):
        err = np.abs(got.double().cpu().numpy() - want)
        assert (err <= 2.0 * u * (bnd + np.abs(want)) + 1e-6).all()
