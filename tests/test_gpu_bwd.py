"""GPU parity of the backward (``attn_bwd``) against the oracle's gradients of
the attention definition.

The forward runs on the GPU (its o and lse feed the backward, as in use); the
oracle computes dQ, dK, dV in fp64 from q, k, v and dO alone.  Tolerance, per
element, from the arithmetic of the GPU path: P and dS are rounded to the
16-bit type before their products, Di comes from the 16-bit O, and the results
are rounded once more, so

    |GPU - oracle| <= 2 u (b + |oracle|) + 1e-6

with u the unit roundoff of the type (2^-11 fp16, 2^-8 bf16) and b the
oracle's magnitude bound of each element (``oracle.attention_bwd(...,
bounds=True)``); the factor 2 covers the fp32 accumulations.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import BLOCK_DIAG, CAUSAL, DENSE, make_qkv, make_qkv_far_below_zero

pytestmark = pytest.mark.gpu

U = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


@pytest.fixture(scope="module")
def af():
    import attention_forward_15_gb300 as m
    from attention_forward_15_gb300 import _build_ext
    _build_ext.build()
    m.load_library()
    assert torch.cuda.is_available()
    return m


def _dout(q, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(q.shape, generator=g).to(q.dtype)


def _case(af, B, H, L, D, mask, bs, dt, scale=None, seed=42, qkv=None):
    q, k, v = make_qkv(B, H, L, D, dt, seed=seed) if qkv is None else qkv
    g = _dout(q, seed + 1)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dev = torch.device("cuda", 0)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    o, lse = af.fwd(qd, kd, vd, mask, bs, scale)
    dq, dk, dv = af.bwd(qd, kd, vd, o, lse, gd, mask, bs, scale)
    torch.cuda.synchronize()
    st, det = af.last_device_status(0)
    assert st == 0, f"device status {st} ({det:#x})"
    ref = oracle.attention_bwd(q, k, v, g, mask, bs, float(np.float32(scale)), bounds=True)
    u = U[dt]
    for name, got, want, b in (("dq", dq, ref[0], ref[3]), ("dk", dk, ref[1], ref[4]),
                               ("dv", dv, ref[2], ref[5])):
        gg = got.double().cpu().numpy()
        assert np.isfinite(gg).all(), f"{name}: non-finite"
        err = np.abs(gg - want)
        tol = 2.0 * u * (b + np.abs(want)) + 1e-6
        worst = np.unravel_index(np.argmax(err - tol), err.shape)
        # the widest tolerance relative to the value, so a vacuous bound is visible
        big = np.abs(want) > 1e-3 * np.abs(want).max()
        rel = (tol[big] / np.abs(want[big])).max() if big.any() else float("nan")   # nan: want is all zero
        print(f"bwd {name} B{B} H{H} L{L} D{D} mask{mask}: max err {err.max():.3e}, max tol {tol.max():.3e}, "
              f"max tol/|ref| {rel:.3e}, max err/tol {(err / tol).max():.3f}")
        assert (err <= tol).all(), (f"{name}: max(err - tol) = {(err - tol).max():.3e} at {worst} "
                                    f"(err {err[worst]:.3e}, tol {tol[worst]:.3e}, ref {want[worst]:.3e})")


CASES = [
    # (B, H, L, D, mask, bs, dtype)
    (1, 2, 256, 64, DENSE, 0, torch.float16),
    (2, 2, 384, 64, CAUSAL, 0, torch.bfloat16),
    (1, 2, 512, 64, BLOCK_DIAG, 64, torch.float16),
    (1, 3, 300, 64, DENSE, 0, torch.bfloat16),          # ragged tail
    (1, 2, 256, 128, DENSE, 0, torch.bfloat16),
    (1, 2, 640, 128, CAUSAL, 0, torch.float16),
    (1, 2, 512, 128, BLOCK_DIAG, 256, torch.bfloat16),
    (1, 2, 333, 128, CAUSAL, 0, torch.float16),         # ragged causal
    (1, 2, 512, 64, BLOCK_DIAG, 16, torch.bfloat16),
    (1, 2, 256, 32, CAUSAL, 0, torch.float16),          # padded head dims
    (1, 2, 256, 96, DENSE, 0, torch.bfloat16),
    (1, 2, 256, 256, DENSE, 0, torch.bfloat16),         # D = 256: half-tile ring, dK/dV split
    (1, 2, 384, 256, CAUSAL, 0, torch.float16),
    (1, 2, 512, 256, BLOCK_DIAG, 64, torch.bfloat16),
    (1, 2, 300, 256, CAUSAL, 0, torch.bfloat16),        # ragged
    (2, 1, 256, 200, DENSE, 0, torch.float16),          # padded into the 256 kernel
    (1, 2, 512, 256, BLOCK_DIAG, 256, torch.float16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}L{}D{}m{}bs{}{}".format(
    *c[:6], "f16" if c[6] == torch.float16 else "bf16"))
def test_bwd_all_elements(af, case):
    _case(af, *case)


# Seeded random configurations (drawn once, the same on every run): any head
# dim, L from 1 to 600, each mask with its block sizes, both dtypes, a random
# scale; combinations the chosen cases above do not name.
def _random_cases(seed=20261204, n=12):
    import random
    rnd = random.Random(seed)
    cases = []
    for _ in range(n):
        mask = rnd.choice([DENSE, CAUSAL, BLOCK_DIAG])
        D = 8 * rnd.randint(1, 32)
        if mask == BLOCK_DIAG:
            bs = rnd.choice([1, 4, 16, 32, 64, 128, 256, 384])
            L = bs * rnd.randint(1, max(1, 600 // bs))
        else:
            bs, L = 0, rnd.randint(1, 600)
        dt = rnd.choice([torch.float16, torch.bfloat16])
        cases.append((1, rnd.randint(1, 2), L, D, mask, bs, dt, round(rnd.uniform(0.02, 0.3), 4),
                      rnd.randint(0, 10 ** 6)))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: "B{}H{}L{}D{}m{}bs{}{}s{}".format(
    *c[:6], "f16" if c[6] == torch.float16 else "bf16", c[7]))
def test_bwd_random_configurations(af, case):
    B, H, L, D, mask, bs, dt, scale, seed = case
    _case(af, B, H, L, D, mask, bs, dt, scale=scale, seed=seed)


@pytest.mark.parametrize("sign", [1, -1])
def test_bwd_scores_far_below_zero(af, sign):
    """Every score near -200 and a ragged tail: P comes from lse, and keys past
    L (zero rows) are cut before their p can overflow."""
    q, k, v, scale = make_qkv_far_below_zero(1, 2, 333, 64, torch.float16, sign)
    _case(af, 1, 2, 333, 64, DENSE, 0, torch.float16, scale=scale, qkv=(q, k, v))


def test_bwd_deterministic(af):
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in make_qkv(1, 4, 512, 128, torch.bfloat16, seed=3))
    g = _dout(q.cpu(), 4).to(dev)
    o, lse = af.fwd(q, k, v, CAUSAL)
    a = af.bwd(q, k, v, o, lse, g, CAUSAL)
    b = af.bwd(q, k, v, o, lse, g, CAUSAL)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_in_cuda_graph(af, D):
    """The backward captured in a CUDA graph (its dQ kernel runs on a stream
    forked from the capturing one and joined back) replays to the eager
    result, bit for bit, twice."""
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in make_qkv(2, 4, 384, D, torch.float16, seed=11))
    g = _dout(q.cpu(), 12).to(dev)
    o, lse = af.fwd(q, k, v, CAUSAL)
    ref = af.bwd(q, k, v, o, lse, g, CAUSAL)
    outs = tuple(torch.empty_like(q) for _ in range(3))
    ws = torch.empty(max(16, af.load_library().attn_bwd_workspace_size(2, 4, 384)), dtype=torch.uint8,
                     device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):      # warm-up outside the capture
        af.bwd(q, k, v, o, lse, g, CAUSAL, dq=outs[0], dk=outs[1], dv=outs[2], workspace=ws)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        af.bwd(q, k, v, o, lse, g, CAUSAL, dq=outs[0], dk=outs[1], dv=outs[2], workspace=ws)
    for _ in range(2):
        for t in outs:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize(dev)
        for x, y in zip(outs, ref):
            assert torch.equal(x, y)
    st, _ = af.last_device_status(0)
    assert st == 0


def test_bwd_argument_errors(af):
    dev = torch.device("cuda", 0)
    q = torch.zeros((1, 1, 128, 100), dtype=torch.float16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    with pytest.raises(af.AttnError) as e:
        af.bwd(q, q, q, q, lse, q)                    # head dims are multiples of 8
    assert e.value.status == 4
    q = torch.zeros((1, 1, 128, 64), dtype=torch.float16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    with pytest.raises(af.AttnError) as e:
        af.bwd(q, q, q, q, lse, q, workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.status == 8


@pytest.mark.parametrize("name", ["causal_b2h32l4096d128_bf16", "dense_b4h16l1024d64_f16",
                                  "dense_b1h16l2048d256_bf16"])
def test_bwd_full_size_heads(af, name):
    """The backward of a full-size workload, in one launch sequence as the
    benchmark runs it (the D = 256 workload at L = 2048 instead of 16384, so
    that the oracle's two heads stay within seconds); the first and the last
    head compared element by element with the oracle's gradients of those
    heads."""
    import math as _m
    from attn_inputs import WORKLOADS, Workload
    if name == "dense_b1h16l2048d256_bf16":
        w = Workload(name, 1, 16, 2048, 256, DENSE, torch.bfloat16, 1.0 / _m.sqrt(256))
    else:
        w = WORKLOADS[name]
    q, k, v = make_qkv(w.B, w.H, w.L, w.D, w.dtype, seed=w.seed)
    g = _dout(q, 99)
    dev = torch.device("cuda", 0)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    o, lse = af.fwd(qd, kd, vd, w.mask, w.block_size, w.sm_scale)
    grads = af.bwd(qd, kd, vd, o, lse, gd, w.mask, w.block_size, w.sm_scale)
    torch.cuda.synchronize()
    assert af.last_device_status(0)[0] == 0
    u = U[w.dtype]
    # the two heads side by side, so that the oracle runs them in parallel
    pick = lambda t: torch.cat([t[0:1, 0:1], t[w.B - 1:w.B, w.H - 1:w.H]], dim=1)
    ref = oracle.attention_bwd(pick(q), pick(k), pick(v), pick(g), w.mask, w.block_size,
                               float(np.float32(w.sm_scale)), bounds=True)
    for name_, got, want, bnd in zip(("dq", "dk", "dv"), grads, ref[:3], ref[3:]):
        gg = pick(got.cpu()).double().numpy()
        err = np.abs(gg - want)
        tol = 2.0 * u * (bnd + np.abs(want)) + 1e-6
        assert np.isfinite(gg).all() and (err <= tol).all(), \
            f"{name_}: max(err - tol) = {(err - tol).max():.3e}"
