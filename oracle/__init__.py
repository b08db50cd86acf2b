"""CPU fp64 oracle for the fused attention forward -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and nothing
here imports the product path.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc and marshals arguments through ctypes.
What the oracle computes, with the passages it follows:

* the attended set of row i: dense = every key; causal = keys j <= i
  ("Fused Attention" page, the stage-2 mask ``offs_m >= start_n + offs_n``);
  block-diagonal = keys in the same bs-block as i ("TLX Block Attention" page,
  the diagonal-block definition at its top);
* scores ``sm_scale * q_i . k_j`` for the attended keys, row max ``m``,
  denominator ``l = sum exp(s_j - m)`` starting at 0, output
  ``sum exp(s_j - m) v_j / l`` ("Triton-CUDA Attention" page, online-softmax
  section: the quantities the recurrence converges to);
* ``lse_i = m + ln l`` ("Fused Attention" page, epilogue ``m_i += log(l_i)``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")

DENSE, CAUSAL, BLOCK_DIAG = 0, 1, 2
F16, BF16 = 0, 1

_libs: dict[int, ctypes.CDLL] = {}
_lock = threading.Lock()


def lib_path(mutant: int = 0) -> str:
    name = "libattn_oracle.so" if mutant == 0 else f"libattn_oracle_mutant{mutant}.so"
    return os.path.join(BUILD_DIR, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake mutant) with gcc."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    # -ffp-contract=off: no fused multiply-add, so x86 and Arm give the same bits.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", f"-DORACLE_MUTANT={mutant}",
           SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant in _libs:
            return _libs[mutant]
        lib = ctypes.CDLL(build(mutant))
        lib.attn_oracle.restype = ctypes.c_int
        lib.attn_oracle.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_long, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_long,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.attn_oracle_widen.restype = ctypes.c_double
        lib.attn_oracle_widen.argtypes = [ctypes.c_uint16, ctypes.c_int]
        lib.attn_oracle_widen_e5m2.restype = ctypes.c_double
        lib.attn_oracle_widen_e5m2.argtypes = [ctypes.c_uint8]
        lib.attn_oracle_round_e5m2.restype = ctypes.c_double
        lib.attn_oracle_round_e5m2.argtypes = [ctypes.c_double]
        lib.attn_oracle_fp8v.restype = ctypes.c_int
        lib.attn_oracle_fp8v.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_long, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_long,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.attn_oracle_bwd.restype = ctypes.c_int
        lib.attn_oracle_bwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_long, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.attn_oracle_f64.restype = ctypes.c_int
        lib.attn_oracle_f64.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_long, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p]
        _libs[mutant] = lib
        return lib


def _bits(t) -> tuple[np.ndarray, int]:
    """Raw 16-bit patterns of a CPU fp16/bf16 torch tensor (or a uint16 array)."""
    if isinstance(t, np.ndarray):
        raise TypeError("pass torch tensors (fp16/bf16) so the dtype is known")
    import torch
    if t.dtype == torch.float16:
        dt = F16
    elif t.dtype == torch.bfloat16:
        dt = BF16
    else:
        raise TypeError(f"oracle takes fp16/bf16 inputs, got {t.dtype}")
    a = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return a, dt


def widen(bits: int, dtype: int, mutant: int = 0) -> float:
    return load(mutant).attn_oracle_widen(bits, dtype)


def attention(q, k, v, mask_kind: int, block_size: int = 0, sm_scale: float | None = None,
              rows=None, nthreads: int = 0, mutant: int = 0):
    """fp64 masked attention of fp16/bf16 ``[B,H,L,D]`` CPU tensors.

    ``sm_scale`` is taken as the fp32 value a caller of the GPU library passes
    (``float(np.float32(sm_scale))``), then used in fp64.  ``rows`` selects flat
    row ids ``(b*H + h)*L + i``; the result is then ``[len(rows), D]``.
    Returns ``(O, lse)`` as float64 numpy arrays.
    """
    qb, dt = _bits(q)
    kb, dtk = _bits(k)
    vb, dtv = _bits(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share one dtype")
    if q.dim() != 4 or tuple(q.shape) != tuple(k.shape) or tuple(q.shape) != tuple(v.shape):
        raise ValueError("q, k, v must all be [B,H,L,D]")
    B, H, L, D = (int(x) for x in q.shape)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    scale = float(np.float32(sm_scale))
    if rows is None:
        rp, nrows = None, 0
        O = np.empty((B, H, L, D), dtype=np.float64)
        lse = np.empty((B, H, L), dtype=np.float64)
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        rp, nrows = ra.ctypes.data, int(ra.size)
        O = np.empty((nrows, D), dtype=np.float64)
        lse = np.empty((nrows,), dtype=np.float64)
    rc = load(mutant).attn_oracle(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, dt,
        B, H, L, D, int(mask_kind), int(block_size), scale,
        rp, nrows, O.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected arguments (B={B} H={H} L={L} D={D} "
                         f"mask={mask_kind} bs={block_size})")
    return O, lse


def widen_e5m2(byte: int, mutant: int = 0) -> float:
    return load(mutant).attn_oracle_widen_e5m2(byte)


def round_e5m2(x: float, mutant: int = 0) -> float:
    return load(mutant).attn_oracle_round_e5m2(float(x))


def attention_fp8v(q, k, vt, mask_kind: int, block_size: int = 0, sm_scale: float | None = None,
                   rows=None, nthreads: int = 0, mutant: int = 0):
    """The FP8 P.V variant of the "Fused Attention" page: q, k fp16/bf16
    ``[B,H,L,D]`` CPU tensors, ``vt`` the transposed V as float8 e5m2
    ``[B,H,D,L]`` (a ``torch.uint8`` or ``torch.float8_e5m2`` CPU tensor).
    Returns ``(O, lse, slack)`` as float64 numpy arrays; ``slack`` bounds, per
    row, the change of O when p values that lie within the error bound of a
    single-precision computation of their exponent (dot-product rounding
    included) from an e5m2 rounding tie round to the other neighbour."""
    qb, dt = _bits(q)
    kb, dtk = _bits(k)
    if dt != dtk:
        raise TypeError("q and k must share one dtype")
    B, H, L, D = (int(x) for x in q.shape)
    if tuple(k.shape) != (B, H, L, D) or tuple(vt.shape) != (B, H, D, L):
        raise ValueError("q, k must be [B,H,L,D] and vt [B,H,D,L]")
    import torch
    vb = np.ascontiguousarray(vt.detach().cpu().contiguous().view(torch.uint8).numpy())
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    scale = float(np.float32(sm_scale))
    if rows is None:
        rp, nrows = None, 0
        O = np.empty((B, H, L, D), dtype=np.float64)
        lse = np.empty((B, H, L), dtype=np.float64)
        slack = np.empty((B, H, L), dtype=np.float64)
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        rp, nrows = ra.ctypes.data, int(ra.size)
        O = np.empty((nrows, D), dtype=np.float64)
        lse = np.empty((nrows,), dtype=np.float64)
        slack = np.empty((nrows,), dtype=np.float64)
    rc = load(mutant).attn_oracle_fp8v(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, dt, B, H, L, D, int(mask_kind),
        int(block_size), scale, rp, nrows, O.ctypes.data, lse.ctypes.data, slack.ctypes.data,
        int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return O, lse, slack


def _f64(t) -> np.ndarray:
    """A CPU torch tensor (any float type) or numpy array as contiguous float64."""
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t, dtype=np.float64)
    return np.ascontiguousarray(t.detach().cpu().double().numpy())


def attention_f64(q, k, v, mask_kind: int, block_size: int = 0, sm_scale: float = 1.0, mutant: int = 0):
    """The forward on fp64 ``[B,H,L,D]`` inputs (no rounding of the inputs):
    returns ``(O, lse)``."""
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    B, H, L, D = qa.shape
    O = np.empty_like(qa)
    lse = np.empty((B, H, L))
    rc = load(mutant).attn_oracle_f64(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, B, H, L, D,
                                      int(mask_kind), int(block_size), float(sm_scale),
                                      O.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return O, lse


def attention_bwd(q, k, v, dout, mask_kind: int, block_size: int = 0, sm_scale: float = 1.0,
                  bounds: bool = False, nthreads: int = 0, mutant: int = 0):
    """Gradients ``(dQ, dK, dV)`` of the attention forward for the output
    gradient ``dout``, from the definition, in fp64 (inputs taken exactly as
    given, 16-bit tensors widened).  With ``bounds``, also ``(bQ, bK, bV)``: per
    element, the magnitudes that rounding P and dS to 16 bits and taking the
    row term from a 16-bit O can act on (see ``attn_oracle.c``)."""
    qa, ka, va, ga = _f64(q), _f64(k), _f64(v), _f64(dout)
    if not (qa.shape == ka.shape == va.shape == ga.shape) or qa.ndim != 4:
        raise ValueError("q, k, v, dout must all be [B,H,L,D]")
    B, H, L, D = qa.shape
    dQ, dK, dV = np.empty_like(qa), np.empty_like(qa), np.empty_like(qa)
    bq = bk = bv = None
    if bounds:
        bq, bk, bv = np.empty_like(qa), np.empty_like(qa), np.empty_like(qa)
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = load(mutant).attn_oracle_bwd(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, ga.ctypes.data,
                                      B, H, L, D, int(mask_kind), int(block_size), float(sm_scale),
                                      dQ.ctypes.data, dK.ctypes.data, dV.ctypes.data,
                                      ptr(bq), ptr(bk), ptr(bv), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected arguments")
    return (dQ, dK, dV, bq, bk, bv) if bounds else (dQ, dK, dV)
