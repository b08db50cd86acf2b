"""CPU-only checks of the C ABI: the library loads without a GPU, exports every
function include/attn.h declares, and rejects bad arguments on the host before
any CUDA call.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_15_gb300 import _build_ext
    import attention_forward_15_gb300 as af
    _build_ext.build()
    return af.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = _declared()
    for n in ("attn_fwd", "attn_fwd_work", "attn_status_string", "attn_last_device_status"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in attn.h but not exported"


def test_abi_version(lib):
    assert lib.attn_abi_version() >> 16 == 1


def test_status_strings(lib):
    for s in range(0, 9):
        assert lib.attn_status_string(s)
    assert lib.attn_status_string(99) == b"unknown status"


def _fwd(lib, B=1, H=1, L=256, D=128, mask=0, bs=0, scale=0.1, dtype=0, ptrs=(16, 16, 16, 16), lse=None):
    q, k, v, o = (ctypes.c_void_p(p) if p else None for p in ptrs)
    return lib.attn_fwd(q, k, v, o, lse, B, H, L, D, mask, bs, scale, dtype, None)


def test_host_validation_before_any_cuda_call(lib):
    # every case is rejected on the host: no device is touched
    assert _fwd(lib, D=100) == 4                  # head dims are multiples of 8 ...
    assert _fwd(lib, D=4) == 4
    assert _fwd(lib, D=264) == 4                  # ... from 8 to 256
    assert _fwd(lib, D=0) == 4
    assert _fwd(lib, dtype=2) == 4
    assert _fwd(lib, mask=3) == 4
    assert _fwd(lib, B=-1) == 2
    assert _fwd(lib, L=-5) == 2
    assert _fwd(lib, mask=2, bs=0) == 3
    assert _fwd(lib, mask=2, bs=48) == 3          # 48 does not divide 256
    assert _fwd(lib, mask=2, bs=96, L=384) == 4   # neither a divisor nor a multiple of 128
    assert _fwd(lib, scale=float("nan")) == 8
    assert _fwd(lib, scale=float("inf")) == 8
    assert _fwd(lib, ptrs=(0, 16, 16, 16)) == 1
    assert _fwd(lib, ptrs=(16, 16, 16, 0)) == 1
    assert _fwd(lib, ptrs=(18, 16, 16, 16)) == 5
    assert _fwd(lib, ptrs=(16, 16, 16, 16), lse=ctypes.c_void_p(20)) == 5
    # empty problems are valid and launch nothing (null pointers allowed)
    assert _fwd(lib, L=0, ptrs=(0, 0, 0, 0)) == 0
    assert _fwd(lib, B=0, ptrs=(0, 0, 0, 0)) == 0


def test_fp8v_host_validation(lib):
    """attn_fwd_fp8v rejects its arguments on the host like attn_fwd, plus L not
    a multiple of 16 (V^T rows must be 16-byte strides for TMA)."""
    def f8(B=1, H=1, L=256, D=128, mask=0, bs=0, scale=0.1, dtype=0, ptrs=(16, 16, 16, 16)):
        q, k, vt, o = (ctypes.c_void_p(p) if p else None for p in ptrs)
        return lib.attn_fwd_fp8v(q, k, vt, o, None, B, H, L, D, mask, bs, scale, dtype, None)
    assert f8(L=200) == 4
    assert f8(L=8, ptrs=(0, 0, 0, 0)) == 4
    assert f8(D=100) == 4
    assert f8(mask=2, bs=48) == 3
    assert f8(ptrs=(16, 16, 0, 16)) == 1
    assert f8(ptrs=(16, 16, 24, 16)) == 5
    assert f8(scale=float("nan")) == 8
    assert f8(L=0, ptrs=(0, 0, 0, 0)) == 0


def test_work_counts(lib):
    import attention_forward_15_gb300 as af
    f, b = af.work(4, 16, 1024, 64, af.DENSE)
    assert f == 4 * 64 * 1024 * 1024 * 64 and b == 4 * 64 * 1024 * 64 * 2
    f, _ = af.work(2, 32, 4096, 128, af.CAUSAL)
    assert f == 4 * 128 * (4096 * 4097 // 2) * 64
    f, b = af.work(8, 16, 8192, 128, af.BLOCK_DIAG, 64)
    assert f == 4 * 128 * 8192 * 64 * 128 and b == 4 * 128 * 8192 * 128 * 2


def test_plan_without_device(lib):
    import attention_forward_15_gb300 as af
    p = af.plan(4, 16, 1024, 64, af.DENSE, with_ctas=False)
    assert p["units"] == 4 * 16 * 4 and p["threads"] == 352 and p["smem_bytes"] <= 232448
    p = af.plan(1, 16, 16384, 256, af.DENSE, dtype=__import__("torch").bfloat16, with_ctas=False)
    assert p["units"] == 16 * 128 and p["threads"] == 192


def test_bwd_host_side(lib):
    """attn_bwd's workspace size, work count and host-side argument checks (no
    compute call: every case is rejected, or empty, before any CUDA call)."""
    import attention_forward_15_gb300 as af
    assert lib.attn_bwd_workspace_size(2, 3, 300) == 2 * 6 * 384 * 4     # rows padded to 128
    assert lib.attn_bwd_workspace_size(1, 1, 0) == 0
    assert lib.attn_bwd_workspace_size(-1, 1, 8) == 0
    f, _ = af.bwd_work(2, 4, 512, 64, af.CAUSAL)
    ff, _ = af.work(2, 4, 512, 64, af.CAUSAL)
    assert f == 2.5 * ff

    def b(D=64, L=256, ws=1 << 20, ptr=16, wsp=16, scale=0.1, mask=0, bs=0):
        p = ctypes.c_void_p(ptr) if ptr else None
        w = ctypes.c_void_p(wsp) if wsp else None
        return lib.attn_bwd(p, p, p, p, p, p, p, p, p, w, ws, 1, 1, L, D, mask, bs, scale, 0, None)
    assert b(D=256) == 4                      # no backward kernel past 128
    assert b(D=100) == 4
    assert b(ws=16) == 8                      # workspace too small
    assert b(scale=float("nan")) == 8
    assert b(ptr=0) == 1
    assert b(wsp=0) == 1
    assert b(ptr=24) == 5
    assert b(mask=2, bs=48) == 3
    assert b(L=0, ptr=0, wsp=0) == 0          # empty: nothing to do
