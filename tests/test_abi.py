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


# Argument checks go through the validate-only entry points (attn_fwd_check,
# attn_fwd_fp8v_check, attn_bwd_check): they run the very checks the launching
# entry points run, make no CUDA call and never dereference the pointers, so
# the placeholder addresses below (16, 18, 24, ...) are never touched.

def _chk(lib, B=1, H=1, L=256, D=128, mask=0, bs=0, scale=0.1, dtype=0, ptrs=(16, 16, 16, 16), lse=None):
    q, k, v, o = (ctypes.c_void_p(p) if p else None for p in ptrs)
    return lib.attn_fwd_check(q, k, v, o, lse, B, H, L, D, mask, bs, scale, dtype)


FWD_CASES = [  # (keyword arguments, expected status)
    (dict(D=100), 4),                   # head dims are multiples of 8 ...
    (dict(D=4), 4),
    (dict(D=264), 4),                   # ... from 8 to 256
    (dict(D=0), 4),
    (dict(dtype=2), 4),
    (dict(mask=3), 4),
    (dict(B=-1), 2),
    (dict(L=-5), 2),
    (dict(mask=2, bs=0), 3),
    (dict(mask=2, bs=48), 3),           # 48 does not divide 256
    (dict(mask=2, bs=96, L=384), 4),    # neither a divisor nor a multiple of 128
    (dict(scale=float("nan")), 8),
    (dict(scale=float("inf")), 8),
    (dict(ptrs=(0, 16, 16, 16)), 1),
    (dict(ptrs=(16, 16, 16, 0)), 1),
    (dict(ptrs=(18, 16, 16, 16)), 5),
    (dict(lse=ctypes.c_void_p(20)), 5),
    (dict(L=0, ptrs=(0, 0, 0, 0)), 0),  # empty problems are valid (null pointers allowed)
    (dict(B=0, ptrs=(0, 0, 0, 0)), 0),
    (dict(), 0),                        # arguments that pass
    (dict(D=96, mask=1, dtype=1), 0),
]


def test_host_validation(lib):
    for kw, want in FWD_CASES:
        assert _chk(lib, **kw) == want, kw


def test_launching_entry_points_run_the_same_checks(lib):
    """attn_fwd and attn_fwd_noalloc return what attn_fwd_check returns for
    every rejected case.  Only where no CUDA device exists (so nothing can be
    launched whatever the checks say) are placeholder addresses passed to
    them; with a device present this is covered by the GPU tests, which pass
    real buffers of the right size."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("placeholder addresses go only to the check entry points when a GPU is present")
    for kw, want in FWD_CASES:
        if want == 0 and kw.get("L", 1) != 0 and kw.get("B", 1) != 0:
            continue                    # would pass the checks: not called here
        a = dict(B=1, H=1, L=256, D=128, mask=0, bs=0, scale=0.1, dtype=0, ptrs=(16, 16, 16, 16), lse=None)
        a.update(kw)
        q, k, v, o = (ctypes.c_void_p(p) if p else None for p in a["ptrs"])
        args = (q, k, v, o, a["lse"], a["B"], a["H"], a["L"], a["D"], a["mask"], a["bs"], a["scale"],
                a["dtype"])
        assert lib.attn_fwd(*args, None) == want, kw
        assert lib.attn_fwd_noalloc(*args, None, None) == want, kw


def test_fp8v_host_validation(lib):
    """attn_fwd_fp8v's checks are attn_fwd's plus L a multiple of 16 (V^T rows
    must be 16-byte strides for TMA)."""
    def f8(B=1, H=1, L=256, D=128, mask=0, bs=0, scale=0.1, dtype=0, ptrs=(16, 16, 16, 16)):
        q, k, vt, o = (ctypes.c_void_p(p) if p else None for p in ptrs)
        return lib.attn_fwd_fp8v_check(q, k, vt, o, None, B, H, L, D, mask, bs, scale, dtype)
    assert f8(L=200) == 4
    assert f8(L=8, ptrs=(0, 0, 0, 0)) == 4
    assert f8(D=100) == 4
    assert f8(mask=2, bs=48) == 3
    assert f8(ptrs=(16, 16, 0, 16)) == 1
    assert f8(ptrs=(16, 16, 24, 16)) == 5
    assert f8(scale=float("nan")) == 8
    assert f8(L=0, ptrs=(0, 0, 0, 0)) == 0
    assert f8() == 0


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
    """attn_bwd's workspace size, work count and host-side argument checks
    (through attn_bwd_check: no CUDA call, the pointers never dereferenced)."""
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
        return lib.attn_bwd_check(p, p, p, p, p, p, p, p, p, w, ws, 1, 1, L, D, mask, bs, scale, 0)
    assert b(D=100) == 4
    assert b(ws=16) == 8                      # workspace too small
    assert b(scale=float("nan")) == 8
    assert b(ptr=0) == 1
    assert b(wsp=0) == 1
    assert b(ptr=24) == 5
    assert b(mask=2, bs=48) == 3
    assert b(L=0, ptr=0, wsp=0) == 0          # empty: nothing to do
    assert b() == 0


def test_host_chunking(lib):
    """attn_fwd_host's chunk choice: the chunks cover every head once, stay
    within 16, keep each chunk's lse slice 16-byte aligned, are one chunk for a
    problem too small to pipeline, and several for the copy-bound headline."""
    import attention_forward_15_gb300 as af
    for B, H, L, D, mask, bs in [(4, 16, 1024, 64, 0, 0), (2, 32, 4096, 128, 1, 0), (1, 2, 256, 128, 2, 64),
                                 (8, 16, 8192, 128, 2, 64), (1, 32, 32768, 128, 1, 0),
                                 (1, 16, 16384, 256, 0, 0), (5, 5, 2047, 64, 0, 0), (3, 7, 1001, 64, 1, 0),
                                 (1, 1, 4096, 64, 0, 0), (2, 9, 333, 128, 0, 0), (64, 64, 128, 32, 1, 0)]:
        for sms in (1, 152):
            hc, n = af.host_chunks(B, H, L, D, mask, bs, sms=sms)
            BH = B * H
            assert 1 <= n <= 16 and 1 <= hc <= BH, (B, H, L, D, sms)
            assert (n - 1) * hc < BH <= n * hc
            if n > 1:
                assert (hc * L * 4) % 16 == 0
    assert af.host_chunks(1, 2, 256, 128, 2, 64) == (2, 1)
    assert af.host_chunks(4, 16, 1024, 64, 0)[1] > 1
    assert af.host_chunks(0, 16, 1024, 64, 0) == (0, 0)
    hc, n = ctypes.c_int(), ctypes.c_int()
    assert lib.attn_fwd_host_chunks(1, 1, 256, 64, 0, 0, 0, 0, ctypes.byref(hc), ctypes.byref(n)) == 8
    assert lib.attn_fwd_host_chunks(1, 1, 256, 100, 0, 0, 0, 152, ctypes.byref(hc), ctypes.byref(n)) == 4


def test_host_entry_point_rejections(lib):
    """attn_fwd_host rejects before any copy or launch: attn_fwd's argument
    checks on the device buffers, then a missing host buffer.  An empty
    problem returns at once.  The placeholder addresses reach the launching
    call only where no CUDA device exists, as for attn_fwd above."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("placeholder addresses go only to the check entry points when a GPU is present")
    P = ctypes.c_void_p

    def host(h=(16, 16, 16, 16), d=(16, 16, 16, 16), lse_h=None, lse_d=None, B=1, H=2, L=256, D=64, mask=0,
             bs=0, scale=0.1, dtype=0):
        hq, hk, hv, ho = (P(x) if x else None for x in h)
        dq, dk, dv, do = (P(x) if x else None for x in d)
        return lib.attn_fwd_host(hq, hk, hv, ho, lse_h, dq, dk, dv, do, lse_d, B, H, L, D, mask, bs, scale,
                                 dtype, None)
    assert host(D=100) == 4
    assert host(mask=2, bs=48) == 3
    assert host(scale=float("nan")) == 8
    assert host(d=(16, 0, 16, 16)) == 1
    assert host(d=(16, 16, 24, 16)) == 5
    assert host(h=(16, 16, 16, 0)) == 1
    assert host(h=(0, 16, 16, 16)) == 1
    assert host(lse_h=P(32), lse_d=None) == 1
    assert host(lse_h=P(32), lse_d=P(20)) == 5
    assert host(B=0, h=(0, 0, 0, 0), d=(0, 0, 0, 0)) == 0


def test_fwd_host_refuses_mismatched_inputs():
    """fwd_host checks k and v against q (shape, dtype, layout) before any
    CUDA call: the library copies q's byte count from each of them."""
    import torch
    import attention_forward_15_gb300 as af
    q = torch.zeros((1, 2, 256, 64), dtype=torch.float16)
    with pytest.raises(ValueError):
        af.fwd_host(q, q[:, :, :128].contiguous(), q)
    with pytest.raises(ValueError):
        af.fwd_host(q, q, q[:, :1].contiguous())
    with pytest.raises(TypeError):
        af.fwd_host(q, q.to(torch.bfloat16), q)
    with pytest.raises(ValueError):
        af.fwd_host(q, q.transpose(2, 3), q)
    with pytest.raises(ValueError):
        af.fwd_host(q[0], q[0], q[0])
