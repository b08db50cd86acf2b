"""The allocation-free entry point attn_fwd_noalloc, called through the C ABI,
against the regular attn_fwd on the same inputs, on two calls in a row.

attn_fwd_noalloc serves callers that may not allocate device memory once
they run (a runtime that reserves its whole budget up front, or a framework
whose pool must own all device memory): its status word lives in a fixed
array compiled into the library instead of memory attn_fwd allocates on its
first call.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

from attn_inputs import BLOCK_DIAG, CAUSAL, DENSE, make_qkv

pytestmark = pytest.mark.gpu

TOL_O = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}


@pytest.fixture(scope="module")
def lib():
    import attention_forward_15_gb300 as af
    from attention_forward_15_gb300 import _build_ext
    _build_ext.build()
    lib = af.load_library()
    lib.attn_fwd_noalloc.restype = ctypes.c_int
    lib.attn_fwd_noalloc.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return lib


CASES = [(2, 4, 640, 128, CAUSAL, 0, torch.bfloat16),
         (1, 4, 512, 64, DENSE, 0, torch.float16),
         (1, 2, 512, 256, DENSE, 0, torch.bfloat16),
         (1, 2, 384, 128, BLOCK_DIAG, 64, torch.float16),
         (1, 2, 256, 64, BLOCK_DIAG, 16, torch.bfloat16)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "L{}D{}m{}bs{}".format(c[2], c[3], c[4], c[5]))
def test_noalloc_matches_regular_entry_point(lib, case):
    import attention_forward_15_gb300 as af
    B, H, L, D, mask, bs, dt = case
    dev = torch.device("cuda", 0)
    scale = 1.0 / math.sqrt(D)
    status = torch.zeros(1, dtype=torch.int32).pin_memory()
    for call, seed in enumerate((11, 12)):                # two calls in a row
        q, k, v = (t.to(dev) for t in make_qkv(B, H, L, D, dt, seed=seed))
        o_ref, lse_ref = af.fwd(q, k, v, mask, bs, scale)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, L, D, mask, bs, scale,
                                  af.BF16 if dt == torch.bfloat16 else af.F16,
                                  ctypes.c_void_p(stream), ctypes.c_void_p(status.data_ptr()))
        assert rc == 0, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        eo = (o.double() - o_ref.double()).abs().max().item()
        el = (lse.double() - lse_ref.double()).abs().max().item()
        assert np.isfinite(eo) and eo <= TOL_O[dt], f"call {call}: max|dO| {eo}"
        assert el <= 1e-3, f"call {call}: max|dlse| {el}"


def test_noalloc_rejects_bad_arguments(lib):
    """Calls that must be refused on the host.  The buffers are real device
    allocations of the size each call describes, so that even a call that
    wrongly got through would stay inside memory it owns."""
    dev = torch.device("cuda", 0)
    for (B, H, L, D, mask, bs), want in (((1, 1, 256, 100, DENSE, 0), 4),       # D not a multiple of 8
                                         ((1, 1, 256, 64, BLOCK_DIAG, 48), 3)):  # 48 does not divide 256
        q, k, v, o = (torch.zeros((B, H, L, D), dtype=torch.float16, device=dev) for _ in range(4))
        rc = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None,
                                  B, H, L, D, mask, bs, 0.1, 0, None, None)
        assert rc == want
    torch.cuda.synchronize()
