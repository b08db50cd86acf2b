"""Python binding of the GB300 fused attention forward (``include/attn.h``).

Argument marshalling only: every step of the attention runs in the CUDA
library ``libattn_gb300.so`` (built in-tree by ``_build_ext.build()``).
PyTorch supplies device memory and the current stream.  There is no CPU or
PyTorch fallback: if the library is missing or a call fails, this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import _build_ext

DENSE, CAUSAL, BLOCK_DIAG = 0, 1, 2
F16, BF16 = 0, 1
# head dims with a kernel of their own; any multiple of 8 up to 256 is accepted
# (it runs in the next one up, the extra columns loaded as zeros)
HEAD_DIMS = (64, 128, 256)

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_NULL", 2: "ATTN_ERR_SHAPE", 3: "ATTN_ERR_BLOCK_SIZE",
          4: "ATTN_ERR_UNSUPPORTED", 5: "ATTN_ERR_ALIGN", 6: "ATTN_ERR_CUDA",
          7: "ATTN_ERR_TIMEOUT", 8: "ATTN_ERR_ARG"}

# Every function the C header declares, with its ctypes signature.
_SIGNATURES = {
    "attn_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_work": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_double)] * 2),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_last_device_status": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                               ctypes.POINTER(ctypes.c_uint)]),
    "attn_fwd_plan": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int)] * 4),
    "attn_abi_version": (ctypes.c_int, []),
    "attn_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 10 + [ctypes.c_int] * 6 +
                      [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_fp8v": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                     ctypes.c_int, ctypes.c_void_p]),
    "attn_bwd": (ctypes.c_int, [ctypes.c_void_p] * 10 + [ctypes.c_size_t] + [ctypes.c_int] * 6 +
                 [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 3),
    "attn_fwd_check": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 +
                       [ctypes.c_float, ctypes.c_int]),
    "attn_fwd_fp8v_check": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 +
                            [ctypes.c_float, ctypes.c_int]),
    "attn_bwd_check": (ctypes.c_int, [ctypes.c_void_p] * 10 + [ctypes.c_size_t] + [ctypes.c_int] * 6 +
                       [ctypes.c_float, ctypes.c_int]),
    "attn_fwd_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 +
                         [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "attn_bwd_work": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_double)] * 2),
    "attn_fwd_host_chunks": (ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_int)] * 2),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build_ext.lib_path()
    if not os.path.exists(p):
        raise ImportError(f"CUDA library not built: {p} (run __graft_entry__.build() or "
                          "attention_forward_15_gb300._build_ext.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float16:
        return F16
    if dt == torch.bfloat16:
        return BF16
    raise TypeError(f"q, k, v must be float16 or bfloat16, got {dt}")


def work(B: int, H: int, L: int, D: int, mask_kind: int, block_size: int = 0,
         dtype: torch.dtype = torch.float16) -> tuple[float, float]:
    """(flops, bytes) of one forward: 4*D*attended pairs, and Q/K/V/O bytes."""
    f, b = ctypes.c_double(), ctypes.c_double()
    rc = load_library().attn_fwd_work(B, H, L, D, mask_kind, block_size, _dtype_code(dtype),
                                      ctypes.byref(f), ctypes.byref(b))
    if rc:
        raise AttnError(rc, "attn_fwd_work")
    return f.value, b.value


def plan(B: int, H: int, L: int, D: int, mask_kind: int, block_size: int = 0,
         dtype: torch.dtype = torch.float16, with_ctas: bool = True) -> dict:
    u, c, t, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = load_library().attn_fwd_plan(B, H, L, D, mask_kind, block_size, _dtype_code(dtype),
                                      ctypes.byref(u), ctypes.byref(c) if with_ctas else None,
                                      ctypes.byref(t), ctypes.byref(s))
    if rc:
        raise AttnError(rc, "attn_fwd_plan")
    out = {"units": u.value, "threads": t.value, "smem_bytes": s.value}
    if with_ctas:
        out["ctas"] = c.value
    return out


def host_chunks(B: int, H: int, L: int, D: int, mask_kind: int, block_size: int = 0,
                dtype: torch.dtype = torch.float16, sms: int = 152) -> tuple[int, int]:
    """(heads per chunk, chunks) that ``fwd_host`` pipelines on a device with
    ``sms`` SMs (host arithmetic only)."""
    hc, n = ctypes.c_int(), ctypes.c_int()
    rc = load_library().attn_fwd_host_chunks(B, H, L, D, mask_kind, block_size, _dtype_code(dtype), sms,
                                             ctypes.byref(hc), ctypes.byref(n))
    if rc:
        raise AttnError(rc, "attn_fwd_host_chunks")
    return hc.value, n.value


def last_device_status(device: int = 0) -> tuple[int, int]:
    st, det = ctypes.c_int(), ctypes.c_uint()
    rc = load_library().attn_last_device_status(device, ctypes.byref(st), ctypes.byref(det))
    if rc:
        raise AttnError(rc, "attn_last_device_status")
    return st.value, det.value


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask_kind: int = DENSE,
        block_size: int = 0, sm_scale: float | None = None, return_lse: bool = True,
        out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
        stream: torch.cuda.Stream | None = None):
    """Fused attention forward of CUDA tensors q, k, v: [B, H, L, D], fp16/bf16.

    Returns ``(o, lse)`` (``lse`` is None when ``return_lse`` is False); the
    call is asynchronous on ``stream`` (default: the current stream).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, L, D]")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, L, D]")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must have the same shape")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k and v must share one dtype")
    if q.device != k.device or q.device != v.device:
        raise ValueError("q, k and v must be on one device")
    B, H, L, D = (int(x) for x in q.shape)
    dt = _dtype_code(q.dtype)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty_like(q)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or o.device != q.device:
        raise ValueError("out must be a contiguous tensor like q")
    lse = None
    if return_lse:
        lse = lse_out if lse_out is not None else torch.empty((B, H, L), dtype=torch.float32,
                                                              device=q.device)
        if (tuple(lse.shape) != (B, H, L) or lse.dtype != torch.float32 or not lse.is_contiguous()
                or lse.device != q.device):
            raise ValueError("lse_out must be a contiguous float32 [B, H, L] tensor on q's device")
    with torch.cuda.device(q.device):
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        rc = load_library().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr() if lse is not None else None,
                                     B, H, L, D, int(mask_kind), int(block_size), float(sm_scale),
                                     dt, ctypes.c_void_p(s.cuda_stream))
    if rc:
        raise AttnError(rc, "attn_fwd")
    return o, lse


def fwd_fp8v(q: torch.Tensor, k: torch.Tensor, vt: torch.Tensor, mask_kind: int = DENSE,
             block_size: int = 0, sm_scale: float | None = None, out: torch.Tensor | None = None,
             lse_out: torch.Tensor | None = None, return_lse: bool = True):
    """``attn_fwd_fp8v``: the FP8 P.V variant.  q, k are fp16/bf16 ``[B,H,L,D]``
    CUDA tensors; ``vt`` is V transposed, ``[B,H,D,L]``, as ``torch.float8_e5m2``
    (or its bytes as ``torch.uint8``).  Returns ``(o, lse)`` like ``fwd``."""
    lib = load_library()
    for t in (q, k, vt):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("fwd_fp8v takes contiguous CUDA tensors")
    B, H, L, D = (int(x) for x in q.shape)
    if tuple(k.shape) != (B, H, L, D) or tuple(vt.shape) != (B, H, D, L):
        raise ValueError("q, k must be [B,H,L,D] and vt [B,H,D,L]")
    if vt.element_size() != 1:
        raise ValueError("vt must be float8 e5m2 (or its uint8 bytes)")
    if k.dtype != q.dtype or k.device != q.device or vt.device != q.device:
        raise ValueError("q, k (one dtype) and vt must be on one device")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty_like(q)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or o.device != q.device:
        raise ValueError("out must be a contiguous tensor like q")
    lse = (lse_out if lse_out is not None else
           torch.empty((B, H, L), dtype=torch.float32, device=q.device)) if return_lse else None
    if lse is not None and (tuple(lse.shape) != (B, H, L) or lse.dtype != torch.float32
                            or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse_out must be a contiguous float32 [B, H, L] tensor on q's device")
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device)
        rc = lib.attn_fwd_fp8v(q.data_ptr(), k.data_ptr(), vt.data_ptr(), o.data_ptr(),
                               lse.data_ptr() if lse is not None else None, B, H, L, D,
                               int(mask_kind), int(block_size), float(sm_scale), _dtype_code(q.dtype),
                               ctypes.c_void_p(s.cuda_stream))
    if rc:
        raise AttnError(rc, "attn_fwd_fp8v")
    return o, lse


def fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask_kind: int = DENSE,
             block_size: int = 0, sm_scale: float | None = None, device: int = 0,
             staging: dict | None = None, return_lse: bool = True):
    """Forward of HOST tensors through ``attn_fwd_host``: the library copies q,
    k, v to the GPU, runs the forward on the current stream of ``device``,
    copies o and lse back and synchronises, pipelined over chunks of heads
    (``host_chunks``) so that both copy directions and the kernels overlap.
    ``staging`` keeps the device buffers (``q_d, k_d, v_d, o_d, lse_d``) and the
    page-locked host outputs (``o_h, lse_h``) for reuse by later calls of the
    same shape, dtype and device (a call with others replaces them).  The
    returned host tensors are those buffers: a later call with the same
    ``staging`` overwrites them.  Returns ``(o_host, lse_host)``."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.device.type != "cpu" or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"fwd_host takes contiguous [B, H, L, D] host tensors ({name})")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    B, H, L, D = (int(x) for x in q.shape)
    dt = _dtype_code(q.dtype)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    # staging buffers are reused only for the shape, dtype and device they were
    # made for; any other call replaces them
    st = staging if staging is not None else {}
    key = (B, H, L, D, q.dtype, int(device))
    if st.get("_key") != key:
        dev = torch.device("cuda", device)
        for name in ("q_d", "k_d", "v_d", "o_d"):
            st[name] = torch.empty(q.shape, dtype=q.dtype, device=dev)
        st["lse_d"] = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        st["o_h"] = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        st["lse_h"] = torch.empty((B, H, L), dtype=torch.float32, pin_memory=True)
        st["_key"] = key
    dev = st["q_d"].device
    with torch.cuda.device(dev):
        s = torch.cuda.current_stream(dev)
        rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), st["o_h"].data_ptr(),
                               st["lse_h"].data_ptr() if return_lse else None,
                               st["q_d"].data_ptr(), st["k_d"].data_ptr(), st["v_d"].data_ptr(),
                               st["o_d"].data_ptr(), st["lse_d"].data_ptr(), B, H, L, D,
                               int(mask_kind), int(block_size), float(sm_scale),
                               dt, ctypes.c_void_p(s.cuda_stream))
    if rc:
        raise AttnError(rc, "attn_fwd_host")
    return st["o_h"], (st["lse_h"] if return_lse else None)


def fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                lse: torch.Tensor | None, mask_kind: int = DENSE, block_size: int = 0,
                sm_scale: float | None = None, status_out: torch.Tensor | None = None):
    """``attn_fwd_noalloc``: the forward for callers that may not allocate
    device memory once they are running (the library's own status word lives
    in a fixed array compiled into it).  The caller passes every buffer,
    including ``o`` and ``lse``; ``status_out`` is an optional pinned host
    uint32/int32 tensor of one element that receives this call's device status
    once the current stream is synchronised.  The first call on a device does
    a one-time set-up and should come before any stream capture."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA [B, H, L, D] tensor")
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise ValueError(f"{name} must match q in shape, dtype and device")
    B, H, L, D = (int(x) for x in q.shape)
    if lse is not None and (tuple(lse.shape) != (B, H, L) or lse.dtype != torch.float32
                            or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [B, H, L] tensor on q's device")
    if status_out is not None and (status_out.device.type != "cpu" or status_out.numel() < 1
                                   or status_out.element_size() != 4):
        raise ValueError("status_out must be a host tensor of 4-byte elements")
    lib = load_library()
    fn = lib.attn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = _SIGNATURES["attn_fwd"][1] + [ctypes.c_void_p]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device)
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                lse.data_ptr() if lse is not None else None, B, H, L, D, int(mask_kind),
                int(block_size), float(sm_scale), _dtype_code(q.dtype),
                ctypes.c_void_p(s.cuda_stream),
                status_out.data_ptr() if status_out is not None else None)
    if rc:
        raise AttnError(rc, "attn_fwd_noalloc")
    return o, lse


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, mask_kind: int = DENSE, block_size: int = 0, sm_scale: float | None = None,
        dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
        workspace: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None):
    """``attn_bwd``: gradients ``(dq, dk, dv)`` of ``sum(dout * o)`` for the
    forward ``fwd(q, k, v, mask_kind, block_size, sm_scale)`` that returned
    ``(o, lse)``.  All CUDA tensors, contiguous, q/k/v/o/dout [B, H, L, D]
    fp16/bf16 (D a multiple of 8 up to 256), lse float32 [B, H, L].
    Asynchronous on ``stream`` (the dQ kernel runs on a second stream of the
    library, forked from and joined back into ``stream``)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA [B, H, L, D] tensor")
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise ValueError(f"{name} must match q in shape, dtype and device")
    B, H, L, D = (int(x) for x in q.shape)
    if (not lse.is_cuda or tuple(lse.shape) != (B, H, L) or lse.dtype != torch.float32
            or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [B, H, L] tensor on q's device")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    lib = load_library()
    outs = []
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        t = torch.empty_like(q) if t is None else t
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous tensor like q")
        outs.append(t)
    need = int(lib.attn_bwd_workspace_size(B, H, L))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    elif workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on q's device")
    with torch.cuda.device(q.device):
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                          lse.data_ptr(), outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          B, H, L, D, int(mask_kind), int(block_size), float(sm_scale),
                          _dtype_code(q.dtype), ctypes.c_void_p(s.cuda_stream))
    if rc:
        raise AttnError(rc, "attn_bwd")
    return tuple(outs)


def bwd_work(B: int, H: int, L: int, D: int, mask_kind: int, block_size: int = 0,
             dtype: torch.dtype = torch.float16):
    """(flops, bytes) of one attn_bwd (flops = 2.5 x the forward's)."""
    f, b = ctypes.c_double(), ctypes.c_double()
    rc = load_library().attn_bwd_work(B, H, L, D, mask_kind, block_size, _dtype_code(dtype),
                                      ctypes.byref(f), ctypes.byref(b))
    if rc:
        raise AttnError(rc, "attn_bwd_work")
    return f.value, b.value
