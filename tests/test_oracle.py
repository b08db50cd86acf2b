"""Pins for the CPU fp64 oracle: checks against facts that do not come from
the oracle itself (closed forms, special cases that reduce to a textbook or
library routine, brute force on tiny inputs, invariants of softmax attention).

Every pin is a plain function taking an ``attn(q, k, v, mask, bs, scale,
rows=None) -> (O, lse)`` callable.  ``test_pins`` runs them on the real
oracle; ``test_planted_mistakes_are_caught`` builds each planted-mistake
mutant of the oracle (a dropped term, a wrong index, a swapped operand, a wrong
mask, ...) and checks that at least one pin fails for every one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import BLOCK_DIAG, CAUSAL, DENSE, make_qkv

TOL = 1e-12


def _attn_for(mutant=0):
    def attn(q, k, v, mask, bs, scale, rows=None):
        return oracle.attention(q, k, v, mask, bs, scale, rows=rows, nthreads=2, mutant=mutant)
    return attn


def _ints(shape, lo, hi, seed, dtype=torch.float16):
    """Small integers (exact in fp16 and bf16) for pins that need exact sums."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(dtype)


def _mask_matrix(L, mask, bs):
    """The attended set written out directly from its definition."""
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    if mask == DENSE:
        return torch.ones(L, L, dtype=torch.bool)
    if mask == CAUSAL:
        return j <= i
    return (j // bs) == (i // bs)


def _torch_ref(q, k, v, mask, bs, scale):
    """Library special case: torch CPU fp64 softmax / logsumexp on the full matrix."""
    qd, kd, vd = q.double(), k.double(), v.double()
    s = torch.matmul(qd, kd.transpose(-1, -2)) * float(np.float32(scale))
    s = s.masked_fill(~_mask_matrix(q.shape[2], mask, bs), float("-inf"))
    return (torch.softmax(s, dim=-1) @ vd).numpy(), torch.logsumexp(s, dim=-1).numpy()


# ----------------------------------------------------------------------------- pins

def pin_torch_library(attn):
    for mask, bs in [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 8), (BLOCK_DIAG, 5)]:
        for dt in (torch.float16, torch.bfloat16):
            L = 40
            q, k, v = make_qkv(2, 2, L, 24, dt, seed=7 + mask)
            O, lse = attn(q, k, v, mask, bs, 0.3)
            Ot, lt = _torch_ref(q, k, v, mask, bs, 0.3)
            assert np.abs(O - Ot).max() < TOL, (mask, bs, dt)
            assert np.abs(lse - lt).max() < TOL, (mask, bs, dt)


def _brute_row(qi, K, V, idx, scale):
    """Pure-Python softmax attention of one row over the key indices idx."""
    s = [scale * math.fsum(a * b for a, b in zip(qi, K[j])) for j in idx]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    l = math.fsum(w)
    o = [math.fsum(w[t] * V[j][d] for t, j in enumerate(idx)) / l for d in range(len(V[0]))]
    return o, m + math.log(l)


def pin_brute_force(attn):
    for mask, bs in [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 3), (BLOCK_DIAG, 1)]:
        L, D = 12, 8
        q, k, v = make_qkv(1, 2, L, D, torch.float16, seed=3)
        scale = float(np.float32(0.41))
        O, lse = attn(q, k, v, mask, bs, scale)
        for h in range(2):
            Q = q[0, h].double().tolist()
            K = k[0, h].double().tolist()
            V = v[0, h].double().tolist()
            for i in range(L):
                if mask == DENSE:
                    idx = list(range(L))
                elif mask == CAUSAL:
                    idx = list(range(i + 1))
                else:
                    idx = list(range((i // bs) * bs, (i // bs + 1) * bs))
                o, ls = _brute_row(Q[i], K, V, idx, scale)
                assert np.abs(O[0, h, i] - np.array(o)).max() < TOL, (mask, h, i)
                assert abs(lse[0, h, i] - ls) < TOL, (mask, h, i)


def pin_brute_force_page_selfcheck(attn):
    """Brute force on the full self-check shape of the TLX Block Attention page
    (B=1, H=2, N=256, D=128, block 64, fp16, N(0,1), seed 42), sampled rows."""
    q, k, v = make_qkv(1, 2, 256, 128, torch.float16, seed=42)
    scale = float(np.float32(1.0 / math.sqrt(128)))
    O, lse = attn(q, k, v, BLOCK_DIAG, 64, scale)
    for h in range(2):
        Q = q[0, h].double().tolist()
        K = k[0, h].double().tolist()
        V = v[0, h].double().tolist()
        for i in (0, 1, 63, 64, 100, 191, 192, 255):
            idx = list(range((i // 64) * 64, (i // 64 + 1) * 64))
            o, ls = _brute_row(Q[i], K, V, idx, scale)
            assert np.abs(O[0, h, i] - np.array(o)).max() < TOL
            assert abs(lse[0, h, i] - ls) < TOL


def pin_hand_example(attn):
    """Closed form: q0=(1,0), keys k_j=(j,0), values v0=(1,0), v1=(0,1), v2=(0,0),
    sm_scale=1.  Scores of row 0 are 0, 1, 2, so the weights are
    1 : e : e^2 and lse = ln(1 + e + e^2).  Row 1 has q1=(0,1): every score is 0,
    so the output is the plain mean of the attended values."""
    q = torch.tensor([[1, 0], [0, 1], [1, 0]], dtype=torch.float16).view(1, 1, 3, 2)
    k = torch.tensor([[0, 0], [1, 0], [2, 0]], dtype=torch.float16).view(1, 1, 3, 2)
    v = torch.tensor([[1, 0], [0, 1], [0, 0]], dtype=torch.float16).view(1, 1, 3, 2)
    e = math.e
    z = 1 + e + e * e
    O, lse = attn(q, k, v, DENSE, 0, 1.0)
    assert abs(O[0, 0, 0, 0] - 1 / z) < TOL and abs(O[0, 0, 0, 1] - e / z) < TOL
    assert abs(lse[0, 0, 0] - math.log(z)) < TOL
    assert abs(O[0, 0, 1, 0] - 1 / 3) < TOL and abs(O[0, 0, 1, 1] - 1 / 3) < TOL
    assert abs(lse[0, 0, 1] - math.log(3)) < TOL
    O, lse = attn(q, k, v, CAUSAL, 0, 1.0)
    assert O[0, 0, 0, 0] == 1 and O[0, 0, 0, 1] == 0 and lse[0, 0, 0] == 0
    assert abs(O[0, 0, 1, 0] - 0.5) < TOL and abs(O[0, 0, 1, 1] - 0.5) < TOL
    assert abs(lse[0, 0, 1] - math.log(2)) < TOL
    # row 2 = row 0 under causal (it sees all three keys)
    assert abs(O[0, 0, 2, 1] - e / z) < TOL and abs(lse[0, 0, 2] - math.log(z)) < TOL


def pin_block_size_L_is_dense(attn):
    q, k, v = make_qkv(1, 3, 48, 16, torch.bfloat16, seed=11)
    O1, l1 = attn(q, k, v, BLOCK_DIAG, 48, 0.25)
    O2, l2 = attn(q, k, v, DENSE, 0, 0.25)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def pin_block_size_one_is_V(attn):
    q, k, v = make_qkv(2, 1, 20, 8, torch.float16, seed=5)
    scale = float(np.float32(0.7))
    O, lse = attn(q, k, v, BLOCK_DIAG, 1, scale)
    assert np.array_equal(O, v.double().numpy())
    qk = (q.double() * k.double()).sum(-1).numpy()
    assert np.abs(lse - scale * qk).max() < TOL


def pin_block_decomposition(attn):
    bs = 8
    q, k, v = make_qkv(1, 2, 32, 16, torch.float16, seed=13)
    O, lse = attn(q, k, v, BLOCK_DIAG, bs, 0.2)
    for b0 in range(0, 32, bs):
        sl = slice(b0, b0 + bs)
        Os, ls = attn(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                      v[:, :, sl].contiguous(), DENSE, 0, 0.2)
        assert np.abs(O[:, :, sl] - Os).max() < TOL and np.abs(lse[:, :, sl] - ls).max() < TOL


def pin_causal_rows(attn):
    q, k, v = make_qkv(1, 2, 33, 16, torch.bfloat16, seed=17)
    scale = float(np.float32(0.35))
    O, lse = attn(q, k, v, CAUSAL, 0, scale)
    Od, ld = attn(q, k, v, DENSE, 0, scale)
    assert np.array_equal(O[:, :, 0], v[:, :, 0].double().numpy())
    qk0 = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1).numpy()
    assert np.abs(lse[:, :, 0] - scale * qk0).max() < TOL
    assert np.abs(O[:, :, -1] - Od[:, :, -1]).max() < TOL
    assert np.abs(lse[:, :, -1] - ld[:, :, -1]).max() < TOL
    q1, k1, v1 = make_qkv(2, 2, 1, 8, torch.float16, seed=19)
    for mask, bs in [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 1)]:
        O1, _ = attn(q1, k1, v1, mask, bs, scale)
        assert np.array_equal(O1, v1.double().numpy())


def _attended_count(L, mask, bs):
    return _mask_matrix(L, mask, bs).sum(-1).numpy()


def pin_constant_keys(attn):
    """All keys equal to kbar: every attended score of a row is the same, so
    O_i is the plain mean of the attended V rows and lse_i = s q_i.kbar + ln|A(i)|."""
    L, D = 24, 8
    for mask, bs in [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 6)]:
        q = _ints((1, 2, L, D), -3, 3, seed=23)
        kbar = _ints((1, 2, 1, D), -2, 2, seed=29)
        k = kbar.expand(1, 2, L, D).contiguous()
        v = _ints((1, 2, L, D), -8, 8, seed=31)
        O, lse = attn(q, k, v, mask, bs, 0.125)
        M = _mask_matrix(L, mask, bs).double()
        mean = (M @ v.double()) / M.sum(-1, keepdim=True)
        assert np.abs(O - mean.numpy()).max() < TOL, mask
        qk = (q.double() * kbar.double()).sum(-1).numpy()
        expect = 0.125 * qk + np.log(_attended_count(L, mask, bs))
        assert np.abs(lse - expect).max() < TOL, mask


def pin_shift_and_affine(attn):
    """K + 1 u^T leaves O unchanged and shifts lse_i by s q_i.u;
    V -> a V + b maps O -> a O + b."""
    L, D = 20, 8
    for mask, bs in [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 4)]:
        q = _ints((1, 1, L, D), -3, 3, seed=37)
        k = _ints((1, 1, L, D), -3, 3, seed=41)
        v = _ints((1, 1, L, D), -6, 6, seed=43)
        u = _ints((1, 1, 1, D), -2, 2, seed=47)
        O, lse = attn(q, k, v, mask, bs, 0.25)
        O2, lse2 = attn(q, (k + u).contiguous(), v, mask, bs, 0.25)
        shift = 0.25 * (q.double() * u.double()).sum(-1).numpy()
        assert np.abs(O2 - O).max() < 1e-11, mask
        assert np.abs(lse2 - (lse + shift)).max() < 1e-11, mask
        O3, lse3 = attn(q, k, (2 * v + 0.5).contiguous(), mask, bs, 0.25)
        assert np.abs(O3 - (2 * O + 0.5)).max() < 1e-11, mask
        assert np.array_equal(lse3, lse)


def pin_bounds(attn):
    """O_i lies in the convex hull of the attended V rows; lse_i lies between
    the row max m and m + ln|A(i)|."""
    L = 30
    for mask, bs in [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 10)]:
        q, k, v = make_qkv(1, 2, L, 16, torch.float16, seed=53)
        O, lse = attn(q, k, v, mask, bs, 0.5)
        M = _mask_matrix(L, mask, bs)
        vd = v.double()[0]
        s = (q.double()[0] @ k.double()[0].transpose(-1, -2)) * 0.5
        for h in range(2):
            for i in range(L):
                rows = vd[h][M[i]]
                assert np.all(O[0, h, i] >= rows.min(0).values.numpy() - TOL)
                assert np.all(O[0, h, i] <= rows.max(0).values.numpy() + TOL)
                m = s[h, i][M[i]].max().item()
                assert m - TOL <= lse[0, h, i] <= m + math.log(int(M[i].sum())) + TOL


def pin_key_permutation(attn):
    q, k, v = make_qkv(1, 2, 26, 16, torch.bfloat16, seed=59)
    perm = torch.randperm(26, generator=torch.Generator().manual_seed(61))
    O, lse = attn(q, k, v, DENSE, 0, 0.3)
    O2, lse2 = attn(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), DENSE, 0, 0.3)
    assert np.abs(O - O2).max() < TOL and np.abs(lse - lse2).max() < TOL


PINS = [pin_torch_library, pin_brute_force, pin_brute_force_page_selfcheck, pin_hand_example,
        pin_block_size_L_is_dense, pin_block_size_one_is_V, pin_block_decomposition,
        pin_causal_rows, pin_constant_keys, pin_shift_and_affine, pin_bounds,
        pin_key_permutation]


# ----------------------------------------------------------------------------- tests

@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pins(pin):
    pin(_attn_for(0))


def test_widen_all_fp16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.widen(int(b), oracle.F16) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_widen_all_bf16_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    want = bits.view(torch.bfloat16).double().numpy()
    got = np.array([oracle.widen(int(b) & 0xFFFF, oracle.BF16) for b in bits.tolist()])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_row_subset_matches_full():
    q, k, v = make_qkv(2, 3, 64, 32, torch.float16, seed=67)
    O, lse = oracle.attention(q, k, v, CAUSAL, 0, 0.2)
    rows = [5, 64 * 3 + 17, 64 * 6 - 1, 0, 64 * 4]
    Or, lr = oracle.attention(q, k, v, CAUSAL, 0, 0.2, rows=rows)
    Of, lf = O.reshape(-1, 32), lse.reshape(-1)
    assert np.array_equal(Or, Of[rows]) and np.array_equal(lr, lf[rows])


def test_rejects_bad_arguments():
    q, k, v = make_qkv(1, 1, 12, 8, torch.float16)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, BLOCK_DIAG, 5, 0.1)       # 5 does not divide 12
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, BLOCK_DIAG, 0, 0.1)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 3, 0, 0.1)


def test_empty_inputs():
    q, k, v = make_qkv(1, 2, 0, 8, torch.float16)
    O, lse = oracle.attention(q, k, v, DENSE, 0, 0.1)
    assert O.shape == (1, 2, 0, 8) and lse.shape == (1, 2, 0)


MUTANTS = {
    1: "causal drops the diagonal",
    2: "sm_scale dropped",
    3: "denominator starts at 1",
    4: "row max dropped from lse",
    5: "wrong row of V",
    6: "strided instead of contiguous blocks",
    7: "K and V swapped",
    8: "log2 in lse",
    9: "row max removed from the denominator only",
    10: "last term of the dot product dropped",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_planted_mistakes_are_caught(mutant):
    attn = _attn_for(mutant)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(attn)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant}: {MUTANTS[mutant]}"


def test_page_fixture_matches_workload_table():
    """The shared input module's copy of the page's test matrix agrees with
    the cited fixture."""
    import json
    import os
    from attn_inputs import PAGE_TEST_MATRIX
    with open(os.path.join(os.path.dirname(__file__), "golden", "page_workloads.json")) as f:
        fx = json.load(f)["fused_attention_test_matrix"]
    names = {torch.float16: "fp16", torch.bfloat16: "bf16"}
    assert [list(c[:4]) + [names[c[4]]] for c in PAGE_TEST_MATRIX] == fx["cases_Z_H_N_D_dtype"]


# ------------------------------------------------------ FP8 P.V variant pins

def _e5m2_values():
    """Every finite non-negative e5m2 value, from the format's definition."""
    vals = []
    for e in range(31):
        for f in range(4):
            vals.append(math.ldexp(f, -16) if e == 0 else math.ldexp(4 + f, e - 17))
    return sorted(set(vals))


def _fp8_pin_top_byte_of_f16(mutant):
    """e5m2 is the upper byte of IEEE binary16: widening byte b equals widening
    the half-precision pattern b << 8."""
    for b in range(256):
        w8 = oracle.widen_e5m2(b, mutant=mutant)
        w16 = oracle.widen(b << 8, oracle.F16, mutant=mutant)
        assert (math.isnan(w8) and math.isnan(w16)) or w8 == w16, (b, w8, w16)


def _fp8_pin_rounding_brute_force(mutant):
    """Rounding to e5m2 is to the nearest value, ties to the even fraction
    (brute force over every value), and saturates at 57344; it agrees with
    torch's float8_e5m2 conversion."""
    vals = _e5m2_values()
    g = np.random.default_rng(3)
    xs = list(np.exp(g.uniform(math.log(1e-6), math.log(5e4), size=400)))
    xs += [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])][::3]        # exact ties
    for x in xs:
        r = oracle.round_e5m2(x, mutant=mutant)
        best = min(abs(v - x) for v in vals)
        assert abs(r - x) == best, (x, r, best)
        cands = [v for v in vals if abs(v - x) == best]
        if len(cands) == 2:                                              # a tie: even fraction
            even = [v for v in cands if (int(v / (math.ldexp(1, math.frexp(v)[1] - 3) if v >= 2 ** -14
                                                   else 2 ** -16)) % 2) == 0]
            assert r in even, (x, r, cands)
        t = float(torch.tensor([x], dtype=torch.float64).to(torch.float8_e5m2).double())
        assert r == t, (x, r, t)
    assert oracle.round_e5m2(60000.0, mutant=mutant) == 57344.0


def _fp8_run(mutant, q, k, vt, mask=DENSE, bs=0, scale=1.0):
    return oracle.attention_fp8v(q, k, vt, mask, bs, scale, nthreads=2, mutant=mutant)


def _fp8_pin_uniform_scores(mutant):
    """Q = 0: every p is exactly 1 (exact in e5m2), so O is the plain mean of
    the attended V rows and lse = ln(number attended), for every mask."""
    B, H, L, D = 1, 2, 256, 8
    g = torch.Generator().manual_seed(4)
    q = torch.zeros(B, H, L, D, dtype=torch.float16)
    k = torch.randn(B, H, L, D, generator=g).to(torch.float16)
    vt = (torch.randn(B, H, D, L, generator=g) * 2).to(torch.float8_e5m2)
    v = vt.double().transpose(-1, -2)                                     # [B,H,L,D]
    for mask, bs in ((DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 64)):
        O, lse, _ = _fp8_run(mutant, q, k, vt, mask, bs)
        M = _mask_matrix(L, mask, bs).double()
        n = M.sum(1)
        want = torch.einsum("ij,bhjd->bhid", M, v) / n[None, None, :, None]
        assert np.abs(O - want.numpy()).max() <= 1e-12
        assert np.abs(lse - np.log(n.numpy())[None, None]).max() <= 1e-12


def _fp8_pin_rounded_weights(mutant):
    """Two keys, scores 0 and -0.05: p = (1, e^-0.05 = 0.951), rounded to e5m2
    (1, 1); O = (1 v0 + 1 v1) / (1 + 0.951) -- the denominator sums the
    unrounded p (the page's l_ij = sum(p))."""
    q = torch.ones(1, 1, 2, 1, dtype=torch.float16)
    k = torch.tensor([0.0, -0.05], dtype=torch.float16).view(1, 1, 2, 1)
    vt = torch.tensor([2.0, 4.0]).to(torch.float8_e5m2).view(1, 1, 1, 2)
    O, lse, _ = _fp8_run(mutant, q, k, vt)
    s1 = float(k[0, 0, 1, 0])
    p1 = math.exp(s1)
    p1r = float(torch.tensor([p1], dtype=torch.float64).to(torch.float8_e5m2).double())
    want = (1.0 * 2.0 + p1r * 4.0) / (1.0 + p1)
    assert p1r == 1.0
    for r in range(2):
        assert abs(O[0, 0, r, 0] - want) <= 1e-12, (O[0, 0, r, 0], want)
        assert abs(lse[0, 0, r] - math.log(1.0 + p1)) <= 1e-12


def _fp8_pin_running_max_across_tiles(mutant):
    """The page rounds P against the running max of the key tiles seen so far:
    key 0 (tile 0, score 0) gets p = 1 when its tile is processed and is only
    rescaled afterwards by exp(0 - 0.6), while the definition (max over all keys
    first) would round e^-0.6 = 0.549 to 0.5.  Every other key scores -30
    (p < 2^-17, rounded to 0)."""
    L = 256
    q = torch.ones(1, 1, L, 1, dtype=torch.float16)
    kk = torch.full((L,), -30.0)
    kk[0] = 0.0
    kk[128] = 0.6
    k = kk.to(torch.float16).view(1, 1, L, 1)
    vv = torch.zeros(L)
    vv[0], vv[128] = 2.0, 8.0
    vt = vv.to(torch.float8_e5m2).view(1, 1, 1, L)
    O, _, _ = _fp8_run(mutant, q, k, vt)
    s128 = float(k[0, 0, 128, 0])
    a = math.exp(0.0 - s128)
    tiny = (L - 2) * math.exp(-30.0 - s128)
    want = (a * 1.0 * 2.0 + 1.0 * 8.0) / (a + 1.0 + tiny)
    assert abs(O[0, 0, 0, 0] - want) <= 1e-9, (O[0, 0, 0, 0], want)


# The oracle's per-row ``slack`` widens the FP8 parity tolerance, so it is
# pinned from above as well as from below: it is zero where no p lies near an
# e5m2 rounding tie, it is exactly one tie's worth where one p sits on a tie,
# and on random inputs it stays under a closed-form bound the test computes
# from its own scores.

def _e5m2_quantum(p: float) -> float:
    """Spacing of float8 e5m2 values around p (2 fraction bits; subnormal
    spacing 2^-16 below 2^-14), from the format's definition."""
    if p < 2.0 ** -14:
        return 2.0 ** -16
    return 2.0 ** (math.floor(math.log2(p)) - 2)


def _split_score_keys(targets):
    """fp16 key rows [x, r] whose scores x + r (with q = [1, 1], scale 1) hit
    ln(target) to about 1e-6: x is the nearest fp16 and r the fp16 residual."""
    rows = []
    for t in targets:
        z = math.log(t)
        x = float(torch.tensor(z, dtype=torch.float16))
        r = float(torch.tensor(z - x, dtype=torch.float16))
        rows.append((x, r))
    return rows


def _fp8_pin_slack_zero_off_ties(mutant):
    """No p near a tie, so no rounding decision is in doubt and slack is 0:
    (a) Q = 0, every p exactly 1; (b) keys whose p lie 0.008 to 0.016 of a
    quantum from the midpoint between two e5m2 neighbours -- far outside the
    single-precision error of the exponent (below 1e-6 relative here, plus 5e-5
    for an approximate exponential, i.e. under 4e-4 of a quantum)."""
    B, H, L, D = 1, 2, 256, 8
    g = torch.Generator().manual_seed(4)
    q = torch.zeros(B, H, L, D, dtype=torch.float16)
    k = torch.randn(B, H, L, D, generator=g).to(torch.float16)
    vt = (torch.randn(B, H, D, L, generator=g) * 2).to(torch.float8_e5m2)
    for mask, bs in ((DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 64)):
        _, _, slack = _fp8_run(mutant, q, k, vt, mask, bs)
        assert (slack == 0.0).all(), slack.max()
    # (b): midpoints (n + 1/2) qv of the binades [1/16, 1), each missed by
    # 0.012 of a quantum on either side
    targets = []
    for e in range(-4, 0):
        qv = 2.0 ** (e - 2)
        for n in range(4, 8):
            for side in (-1, 1):
                targets.append((n + 0.5 + side * 0.012) * qv)
    keys = [(0.0, 0.0)] + _split_score_keys(targets)       # key 0: score 0, the row max
    L = len(keys)
    kk = torch.tensor(keys, dtype=torch.float16).view(1, 1, L, 2)
    qq = torch.ones(1, 1, L, 2, dtype=torch.float16)
    for x, r in keys[1:]:                                   # the test's own check of each p
        p = math.exp(x + r)
        qv = _e5m2_quantum(p)
        dist = abs(p / qv - math.floor(p / qv) - 0.5)
        assert 0.008 <= dist <= 0.016, (p, dist)
    vt = torch.linspace(-3, 3, 2 * L).view(1, 1, 2, L).to(torch.float8_e5m2)
    _, _, slack = _fp8_run(mutant, qq, kk, vt)
    assert (slack == 0.0).all(), slack.max()


def _fp8_pin_slack_at_exact_tie(mutant):
    """Key 1's p sits on the e5m2 tie 0.9375 (between 0.875 and 1) to about
    1e-6: rounding it either way is correct, and the largest change of an
    element of O that the choice makes is qv max_d |v_1d| / l with qv = 1/8 --
    which is what slack must be, exactly (one key, counted once, by the largest
    element of its V row)."""
    (x, r), = _split_score_keys([0.9375])
    kk = torch.tensor([[0.0, 0.0], [x, r]], dtype=torch.float16).view(1, 1, 2, 2)
    qq = torch.ones(1, 1, 2, 2, dtype=torch.float16)
    p1 = math.exp(x + r)
    assert abs(p1 / 0.9375 - 1.0) <= 2e-6
    v1 = (2.0, -1.5, 0.75)                                 # exact in e5m2
    vt = torch.tensor([[1.0, v1[0]], [0.5, v1[1]], [-1.0, v1[2]]]).to(torch.float8_e5m2).view(1, 1, 3, 2)
    vt = vt.view(torch.uint8)
    kk3 = torch.cat([kk, torch.zeros(1, 1, 2, 1, dtype=torch.float16)], dim=-1)
    qq3 = torch.cat([qq, torch.zeros(1, 1, 2, 1, dtype=torch.float16)], dim=-1)
    _, _, slack = _fp8_run(mutant, qq3, kk3, vt)
    want = 0.125 * max(abs(x) for x in v1) / (1.0 + p1)
    assert np.abs(slack - want).max() <= 1e-12 * want, (slack, want)


def _fp8_pin_slack_closed_form_bound(mutant):
    """Random N(0,1) inputs, one 128-key tile (so the running max is the row
    max): slack <= sum over the keys whose p lies within 2e-4 p (a stated bound
    of the single-precision error of the exponent on these inputs: D 2^-24
    sum|q k| scale is below 4e-5, plus 5e-5 for an approximate exponential) of
    a tie of qv max_d |v_jd| / l, with p, qv, l computed here in fp64 from the
    widened inputs."""
    B, H, L, D = 1, 4, 128, 64
    scale = 0.125
    q, k, v = make_qkv(B, H, L, D, torch.float16, seed=17)
    vt = v.float().to(torch.float8_e5m2).transpose(-1, -2).contiguous()
    _, _, slack = _fp8_run(mutant, q, k, vt, DENSE, 0, scale)
    s = (q.double() @ k.double().transpose(-1, -2)).numpy() * scale
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    l = p.sum(axis=-1)
    vmax = np.abs(vt.double().numpy()).max(axis=-2)                 # [B, H, L] per key
    bound = np.zeros_like(l)
    n_near = 0
    for b in range(B):
        for h in range(H):
            for i in range(L):
                for j in range(L):
                    qv = _e5m2_quantum(p[b, h, i, j])
                    t = p[b, h, i, j] / qv
                    if abs(t - math.floor(t) - 0.5) < 2e-4 * t:
                        bound[b, h, i] += qv * vmax[b, h, j] / l[b, h, i]
                        n_near += 1
    assert (slack <= bound + 1e-15).all(), (slack - bound).max()
    assert n_near < 0.01 * B * H * L * L        # the bound itself is not vacuous


FP8_PINS = [_fp8_pin_top_byte_of_f16, _fp8_pin_rounding_brute_force, _fp8_pin_uniform_scores,
            _fp8_pin_rounded_weights, _fp8_pin_running_max_across_tiles, _fp8_pin_slack_zero_off_ties,
            _fp8_pin_slack_at_exact_tie, _fp8_pin_slack_closed_form_bound]


@pytest.mark.parametrize("pin", FP8_PINS, ids=lambda f: f.__name__)
def test_fp8_pins(pin):
    pin(0)


FP8_MUTANTS = {
    11: "e5m2 rounding truncates",
    12: "denominator sums the rounded p",
    13: "V read untransposed",
    14: "tie band 100x too wide",
    15: "tie counted per column",
}


@pytest.mark.parametrize("mutant", sorted(FP8_MUTANTS), ids=lambda m: FP8_MUTANTS[m].replace(" ", "_"))
def test_fp8_planted_mistakes_are_caught(mutant):
    caught = []
    for pin in FP8_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant}: {FP8_MUTANTS[mutant]}"


# ----------------------------------------------------------------------------- backward pins
# The backward is the gradient of the forward; its pins are facts that do not
# come from the backward code: derivatives taken numerically from the forward,
# a library's automatic differentiation of the same function, and invariants
# of softmax attention.

def _bwd_inputs(seed, L=10, D=6, H=2):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn((1, H, L, D), generator=g, dtype=torch.float64) for _ in range(4))


BWD_MASKS = [(DENSE, 0), (CAUSAL, 0), (BLOCK_DIAG, 5)]


def _bwd_pin_finite_differences(mutant):
    """<dX, E> against the central difference of sum(dO * O(X + eps E)) for a few
    random directions E, X each of q, k, v; the forward is the oracle's own."""
    scale = 0.7
    for mask, bs in BWD_MASKS:
        q, k, v, g = _bwd_inputs(3 + mask)
        dq, dk, dv = oracle.attention_bwd(q, k, v, g, mask, bs, scale, mutant=mutant)
        gn = g.numpy()

        def loss(qq, kk, vv):
            O, _ = oracle.attention_f64(qq, kk, vv, mask, bs, scale, mutant=mutant)
            return float((O * gn).sum())

        rng = np.random.default_rng(11 + mask)
        eps = 1e-6
        for which, grad in ((0, dq), (1, dk), (2, dv)):
            for _ in range(3):
                E = rng.standard_normal(q.shape)
                args_p = [q.numpy(), k.numpy(), v.numpy()]
                args_m = [q.numpy(), k.numpy(), v.numpy()]
                args_p[which] = args_p[which] + eps * E
                args_m[which] = args_m[which] - eps * E
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                an = float((grad * E).sum())
                assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (mask, which, fd, an)


def _bwd_pin_torch_autograd(mutant):
    """Library special case: torch's automatic differentiation of the same
    masked softmax attention (additive -inf mask), fp64."""
    scale = -0.45
    for mask, bs in BWD_MASKS:
        q, k, v, g = _bwd_inputs(30 + mask, L=20, D=8)
        dq, dk, dv = oracle.attention_bwd(q, k, v, g, mask, bs, scale, mutant=mutant)
        qq, kk, vv = (t.clone().requires_grad_() for t in (q, k, v))
        s = (qq @ kk.transpose(-1, -2)) * scale
        s = s.masked_fill(~_mask_matrix(20, mask, bs), float("-inf"))
        (torch.softmax(s, dim=-1) @ vv).backward(g)
        for a, b in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
            assert np.abs(a - b.numpy()).max() <= 1e-10


def _bwd_pin_invariants(mutant):
    """Adding one vector to every key leaves every row's softmax unchanged, so
    the key gradients of a head sum to zero; the weights of a row sum to one,
    so the value gradients of a head sum to the sum of the output gradients."""
    for mask, bs in BWD_MASKS:
        q, k, v, g = _bwd_inputs(50 + mask, L=20, D=5)
        dq, dk, dv = oracle.attention_bwd(q, k, v, g, mask, bs, 0.9, mutant=mutant)
        assert np.abs(dk.sum(axis=2)).max() <= 1e-12
        assert np.abs(dv.sum(axis=2) - g.numpy().sum(axis=2)).max() <= 1e-12


def _bwd_pin_block_size_one(mutant):
    """Block size 1: every row attends only itself with weight 1, so dV = dO
    and the softmax passes no gradient to q or k."""
    q, k, v, g = _bwd_inputs(70, L=12, D=4)
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, BLOCK_DIAG, 1, 0.3, mutant=mutant)
    assert np.abs(dv - g.numpy()).max() == 0.0
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0


# The magnitudes bQ, bK, bV scale the backward's parity tolerance, so they are
# pinned from above: on inputs where the triangle inequality behind them is an
# equality they must equal |dQ|, |dK|, |dV|, and block size 1 gives each in
# closed form.

def _bwd_pin_bound_of_dv_is_tight(mutant):
    """dO >= 0 everywhere: every term P[i,j] dO[i,d] of dV[j,d] is >= 0, so
    bV = sum_i P[i,j] |dO[i,d]| equals |dV| exactly (every mask)."""
    for mask, bs in BWD_MASKS:
        q, k, v, g = _bwd_inputs(110 + mask, L=15, D=5)
        g = g.abs()
        _, _, dv, _, _, bv = oracle.attention_bwd(q, k, v, g, mask, bs, 0.8, bounds=True, mutant=mutant)
        assert np.abs(bv - np.abs(dv)).max() <= 1e-12 * max(1.0, np.abs(dv).max())


def _bwd_pin_bounds_tight_on_two_keys(mutant):
    """Two keys k = (a, -a), both queries 1 (one head dim), so each row has the
    weights (w, 1 - w), w = 1/(1 + exp(-2 s a)); V = c (1 - w, -w) makes O = 0,
    so the row terms a_i = sum_d |dO O| and D_i vanish and dS[i] = c w (1 - w)
    dO_i (1, -1).  Then dQ_i = 2 s a dS[i,0] with every term of bQ of one sign,
    and with dO = (1, 2) (one sign) the same holds for dK: bQ = |dQ| and
    bK = |dK| exactly, and bV = |dV| (dO >= 0)."""
    for a, scale, c in ((0.7, 0.9, 1.5), (-1.2, 0.4, -0.8), (0.3, -2.0, 2.5)):
        w = 1.0 / (1.0 + math.exp(-2.0 * scale * a))
        q = torch.ones(1, 1, 2, 1, dtype=torch.float64)
        k = torch.tensor([a, -a], dtype=torch.float64).view(1, 1, 2, 1)
        v = torch.tensor([c * (1 - w), -c * w], dtype=torch.float64).view(1, 1, 2, 1)
        g = torch.tensor([1.0, 2.0], dtype=torch.float64).view(1, 1, 2, 1)
        dq, dk, dv, bq, bk, bv = oracle.attention_bwd(q, k, v, g, DENSE, 0, scale, bounds=True, mutant=mutant)
        ds0 = c * w * (1 - w) * np.array([1.0, 2.0])          # dS[i, 0] of rows 0, 1
        assert np.abs(dq.reshape(2) - 2 * scale * a * ds0).max() <= 1e-12
        for x, bx in ((dq, bq), (dk, bk), (dv, bv)):
            assert np.abs(bx - np.abs(x)).max() <= 1e-12 * max(1.0, np.abs(x).max()), (x, bx)


def _bwd_pin_bounds_block_size_one(mutant):
    """Block size 1: P = 1 on the diagonal, dS = 0, O_i = v_i, so bV = |dO|,
    bQ[i,d] = |s| a_i |k[i,d]| and bK[i,d] = |s| a_i |q[i,d]| with
    a_i = sum_d |dO[i,d] v[i,d]|."""
    q, k, v, g = _bwd_inputs(120, L=9, D=4)
    scale = -0.7
    _, _, _, bq, bk, bv = oracle.attention_bwd(q, k, v, g, BLOCK_DIAG, 1, scale, bounds=True, mutant=mutant)
    a = (g * v).abs().sum(dim=-1, keepdim=True).numpy()
    assert np.abs(bv - g.abs().numpy()).max() <= 1e-15
    assert np.abs(bq - abs(scale) * a * k.abs().numpy()).max() <= 1e-12
    assert np.abs(bk - abs(scale) * a * q.abs().numpy()).max() <= 1e-12


BWD_PINS = [_bwd_pin_finite_differences, _bwd_pin_torch_autograd, _bwd_pin_invariants,
            _bwd_pin_block_size_one, _bwd_pin_bound_of_dv_is_tight, _bwd_pin_bounds_tight_on_two_keys,
            _bwd_pin_bounds_block_size_one]


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda f: f.__name__)
def test_bwd_pins(pin):
    pin(0)


BWD_MUTANTS = {
    21: "row term Di dropped from dS",
    22: "sm_scale dropped from dK",
    23: "P transposed in dV",
    24: "bound of dQ 4x too large",
    25: "bound of dK 4x too large",
    26: "bound of dV 4x too large",
}


@pytest.mark.parametrize("mutant", sorted(BWD_MUTANTS), ids=lambda m: BWD_MUTANTS[m].replace(" ", "_"))
def test_bwd_planted_mistakes_are_caught(mutant):
    caught = []
    for pin in BWD_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant}: {BWD_MUTANTS[mutant]}"


def test_bwd_bounds_dominate_gradients():
    """The magnitude outputs bound what they describe: |dV| <= bV, and bK, bQ
    are at least |dK|, |dQ| (triangle inequality)."""
    q, k, v, g = _bwd_inputs(90, L=24, D=8)
    dq, dk, dv, bq, bk, bv = oracle.attention_bwd(q, k, v, g, CAUSAL, 0, 0.6, bounds=True)
    assert (np.abs(dv) <= bv + 1e-12).all()
    assert (np.abs(dk) <= bk + 1e-12).all() and (np.abs(dq) <= bq + 1e-12).all()
