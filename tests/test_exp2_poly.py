"""The FMA-pipe exp2 used for part of the softmax exponentials: its
coefficients in the kernel are the ones the committed Remez fit produces, and
the whole fp32 evaluation (range reduction + Horner, mirrored in numpy) stays
within 1e-4 relative error of exp2 — below the rounding of P to fp16 (4.9e-4)
or bf16 (3.9e-3)."""
import importlib.util
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "attention_forward_15_gb300", "csrc")


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", os.path.join(CSRC, "fit_exp2_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _kernel_coeffs():
    src = open(os.path.join(CSRC, "attn_fwd_kernel.cuh")).read()
    return [float(re.search(rf"\bc{k} = ([0-9.eE+-]+)f", src).group(1)) for k in range(4)]


def test_kernel_coefficients_match_the_fit():
    fit = _fit_module()
    c32 = [float(np.float32(v)) for v in fit.remez_exp2(3)]
    assert np.allclose(_kernel_coeffs(), c32, rtol=1e-6, atol=0)


def test_error_bound():
    fit = _fit_module()
    assert fit.max_rel_error_fp32(_kernel_coeffs()) < 1e-4


def test_special_points():
    fit = _fit_module()
    c = _kernel_coeffs()
    x = np.array([0.0, 1.0, -1.0, 8.0, -20.5, 0.49999997, -0.5], dtype=np.float32)
    rel = np.abs(fit.emulate(x, c) / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() < 1e-4
    # far below the clamp the value is tiny but positive and finite
    tiny = fit.emulate(np.array([-1000.0, -np.inf], dtype=np.float32), c)
    assert np.all(np.isfinite(tiny)) and np.all(tiny >= 0) and np.all(tiny < 1e-37)
