"""``bench.py --shape``: the ad hoc workload a profiler run names is parsed into
the same Workload the named workloads use, and malformed specs are refused."""
import math
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attn_inputs import BLOCK_DIAG, CAUSAL  # noqa: E402


def test_shape_parses_into_a_workload():
    w = bench.shape_workload("1,8,8192,128,causal,bf16")
    assert (w.B, w.H, w.L, w.D, w.mask, w.dtype) == (1, 8, 8192, 128, CAUSAL, torch.bfloat16)
    assert w.block_size == 0 and w.sm_scale == pytest.approx(1 / math.sqrt(128))
    w = bench.shape_workload("2,4,512,64,block_diag,fp16,64")
    assert (w.mask, w.block_size, w.dtype) == (BLOCK_DIAG, 64, torch.float16)
    assert w.name == "block_diag_b2h4l512d64_fp16_bs64"
    # the flop count the bench divides by: attended pairs per head
    assert bench.attended_pairs(w) == 512 * 64


@pytest.mark.parametrize("spec", ["1,8,8192,128,causal", "1,8,8192,128,triangle,bf16",
                                  "1,8,8192,128,causal,fp32", "1,2,256,64,block_diag,fp16",
                                  "1,2,256,64,block_diag,fp16,48", "1,2,256,64,dense,fp16,64"])
def test_malformed_shapes_are_refused(spec):
    with pytest.raises(SystemExit):
        bench.shape_workload(spec)
