"""GPU parity of the FP8 P.V variant (``attn_fwd_fp8v``) against the oracle's
rendering of the page's recurrence (``oracle.attention_fp8v``).

Both sides round P to float8 e5m2 against the same running max, so P agrees
except where a p lies at a rounding tie of e5m2 within single-precision error;
the oracle returns, per row, a bound on what such ties can move (``slack``).
Tolerance per row: that slack plus the 16-bit tolerance of O (4e-3 fp16,
1.6e-2 bf16); lse within 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import BLOCK_DIAG, CAUSAL, DENSE, make_qkv, make_qkv_far_below_zero, make_vt_e5m2

pytestmark = pytest.mark.gpu

TOL_O = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}
TOL_LSE = 1e-3


@pytest.fixture(scope="module")
def af():
    import attention_forward_15_gb300 as m
    from attention_forward_15_gb300 import _build_ext
    _build_ext.build()
    m.load_library()
    assert torch.cuda.is_available()
    return m


def _case(af, B, H, L, D, mask, bs, dt, scale=None, seed=42, std=1.0, rows=None, qkv=None):
    q, k, v = make_qkv(B, H, L, D, dt, seed=seed, std=std) if qkv is None else qkv
    vt = make_vt_e5m2(v)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dev = torch.device("cuda", 0)
    o, lse = af.fwd_fp8v(q.to(dev), k.to(dev), vt.to(dev), mask, bs, scale)
    torch.cuda.synchronize()
    O, LSE, slack = oracle.attention_fp8v(q, k, vt, mask, bs, scale, rows=rows)
    og = o.double().cpu().numpy()
    lg = lse.double().cpu().numpy()
    if rows is not None:
        og = og.reshape(-1, D)[rows]
        lg = lg.reshape(-1)[rows]
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    err = np.abs(og - O).max(axis=-1)
    tol = slack + TOL_O[dt]
    worst = int(np.argmax(err - tol))
    # how much the tie slack widens the tolerance, so a vacuous one is visible
    print(f"fp8v B{B} H{H} L{L} D{D} mask{mask}: max|dO| {err.max():.3e}, max slack {slack.max():.3e}, "
          f"rows with slack {np.mean(slack > 0):.3f}, rows past the 16-bit tolerance "
          f"{np.mean(err > TOL_O[dt]):.4f}")
    assert (err <= tol).all(), f"max|dO| - tol = {(err - tol).max():.3e} (err {err.flat[worst]:.3e})"
    assert np.abs(lg - LSE).max() <= TOL_LSE
    return float(err.max()), float(slack.max())


CASES = [
    # (B, H, L, D, mask, bs, dtype)
    (2, 3, 384, 64, DENSE, 0, torch.float16),
    (1, 2, 400, 64, CAUSAL, 0, torch.bfloat16),          # ragged tail (400 = 16 x 25)
    (1, 2, 512, 64, BLOCK_DIAG, 64, torch.float16),
    (2, 2, 512, 128, DENSE, 0, torch.bfloat16),
    (1, 3, 640, 128, CAUSAL, 0, torch.float16),
    (1, 2, 768, 128, BLOCK_DIAG, 256, torch.bfloat16),
    (1, 2, 512, 256, DENSE, 0, torch.bfloat16),
    (1, 2, 336, 256, CAUSAL, 0, torch.float16),
    (1, 2, 512, 96, DENSE, 0, torch.float16),            # padded head dim
    (1, 2, 256, 32, CAUSAL, 0, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}L{}D{}m{}bs{}{}".format(
    *c[:6], "f16" if c[6] == torch.float16 else "bf16"))
def test_fp8v_all_elements(af, case):
    _case(af, *case)


# Seeded random configurations (drawn once, the same on every run): any head
# dim, L a multiple of 16 up to 800, each mask with its block sizes, both
# dtypes, scales up to 1/sqrt(D) (score spreads within the workloads').
def _random_cases(seed=20261205, n=10):
    import random
    rnd = random.Random(seed)
    cases = []
    for _ in range(n):
        mask = rnd.choice([DENSE, CAUSAL, BLOCK_DIAG])
        D = 8 * rnd.randint(1, 32)
        if mask == BLOCK_DIAG:
            bs = rnd.choice([16, 32, 64, 128, 256])
            L = bs * rnd.randint(1, max(1, 800 // bs))
        else:
            bs, L = 0, 16 * rnd.randint(1, 50)
        dt = rnd.choice([torch.float16, torch.bfloat16])
        scale = round(rnd.uniform(0.3, 1.0) / math.sqrt(D), 5)
        cases.append((1, rnd.randint(1, 2), L, D, mask, bs, dt, scale, rnd.randint(0, 10 ** 6)))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: "B{}H{}L{}D{}m{}bs{}{}s{}".format(
    *c[:6], "f16" if c[6] == torch.float16 else "bf16", c[7]))
def test_fp8v_random_configurations(af, case):
    B, H, L, D, mask, bs, dt, scale, seed = case
    _case(af, B, H, L, D, mask, bs, dt, scale=scale, seed=seed)


def test_fp8v_wide_scores(af):
    """N(0, 2^2) inputs: the running max moves often, so P is rounded against
    many different references and O is rescaled on most rows."""
    _case(af, 1, 2, 512, 128, CAUSAL, 0, torch.float16, std=2.0, scale=0.2)


@pytest.mark.parametrize("D,mask,bs,dt", [(64, CAUSAL, 0, torch.float16), (128, DENSE, 0, torch.bfloat16),
                                         (256, BLOCK_DIAG, 64, torch.float16)])
@pytest.mark.parametrize("sign", [1, -1])
def test_fp8v_scores_far_below_zero(af, D, mask, bs, dt, sign):
    """Every attended score near -200: P is rounded against the row max (about
    -200), so an extreme that let a stray 0 in would round P against 0 and
    underflow it."""
    q, k, v, scale = make_qkv_far_below_zero(1, 2, 384, D, dt, sign)
    _case(af, 1, 2, 384, D, mask, bs, dt, scale=scale, qkv=(q, k, v))


def test_fp8v_full_size_sampled(af):
    """The causal B2 H32 L4096 D128 workload, sampled rows."""
    rows = np.array(sorted(set(int(r) for r in np.random.default_rng(2).integers(0, 2 * 32 * 4096, 160))))
    _case(af, 2, 32, 4096, 128, CAUSAL, 0, torch.bfloat16, rows=rows)


def test_fp8v_argument_errors(af):
    dev = torch.device("cuda", 0)
    q = torch.zeros((1, 1, 200, 64), dtype=torch.float16, device=dev)   # L not a multiple of 16
    vt = torch.zeros((1, 1, 64, 200), dtype=torch.uint8, device=dev)
    with pytest.raises(af.AttnError) as e:
        af.fwd_fp8v(q, q, vt)
    assert e.value.status == 4
    q = torch.zeros((1, 1, 0, 64), dtype=torch.float16, device=dev)
    vt = torch.zeros((1, 1, 64, 0), dtype=torch.uint8, device=dev)
    o, lse = af.fwd_fp8v(q, q, vt)
    assert o.shape == q.shape
