"""The seeded synthetic workloads: shapes, FLOPs and value distributions.

The GEMM sizes are fixed by the workload descriptions (FP8 per-tensor
128x1024x1024; W4A16 decode M {1,16,64} on three (K,N); the FP8 DiT MLP at
M = 4096*B; MXFP8 at M = 20280; the mixed stack of 4 NVFP4 attention and 4
FP8 MLP linears at M = 32768), so their FLOP counts are checked against the
values that follow from them.  The activations with outlier channels have
ceil(1% of K) columns replaced by 20 * Student-t(3); the rest is N(0, 1).
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from serving_amax_reduce_gb300 import inputs  # noqa: E402


def tflop(lins):
    return sum(lin.flops() for lin in lins) / 1e12


def test_workload_gemm_sizes_and_flops():
    lins = bench.workload_linears()
    by = {}
    for group, lin in lins:
        by.setdefault(group, []).append(lin)
    assert [len(by[g]) for g in ("fp8_tensor", "w4a16", "fp8_block", "mxfp8", "mixed")] == [1, 9, 6, 3, 8]
    assert by["fp8_tensor"][0].flops() == 2 * 128 * 1024 * 1024            # 0.268 GFLOP
    fp8_block = sorted(round(lin.flops() / 1e12, 3) for lin in by["fp8_block"])
    assert fp8_block == [0.309, 0.309, 1.237, 1.237, 2.474, 2.474]
    assert sorted(round(lin.flops() / 1e12, 3) for lin in by["mxfp8"]) == [1.063, 2.871, 2.871]
    assert round(tflop(by["mixed"]), 2) == 12.37
    assert sorted((lin.M, lin.K, lin.N) for lin in by["w4a16"]) == sorted(
        (M, K, N) for (K, N) in [(4096, 4096), (4096, 12288), (12288, 4096)] for M in (1, 16, 64))
    # the ragged row tail of the video-DiT shape
    assert all(lin.M == 20280 and lin.M % 128 == 56 for lin in by["mxfp8"])
    # the mixed stack: q, k, v, out at d x d in NVFP4; two up and two down MLP linears in FP8 block-128
    mixed = [(lin.w_fmt, lin.K, lin.N) for lin in by["mixed"]]
    assert mixed[:4] == [("nvfp4", 3072, 3072)] * 4
    assert sorted(mixed[4:]) == [("fp8_block128", 3072, 12288)] * 2 + [("fp8_block128", 12288, 3072)] * 2


def test_next_rows_reuse_the_workload_shapes():
    lins = dict()
    for group, lin in bench.workload_linears(next_rows=True):
        lins.setdefault(group, []).append(lin)
    assert sorted((lin.K, lin.N, lin.M) for lin in lins["mxfp4"]) == sorted(
        (K, N, 20280) for (K, N) in inputs.MXFP8_SHAPES)
    for g in ("fp8_group", "int8"):
        assert sorted((lin.K, lin.N, lin.M) for lin in lins[g]) == sorted(
            (K, N, 4096) for (K, N) in inputs.FP8_MLP_SHAPES)
    assert [(lin.M, lin.K, lin.N) for lin in lins["fp8_tensor_fused"]] == [(128, 1024, 1024)]
    assert sorted((lin.K, lin.N, lin.M) for lin in lins["mxfp4_dual"]) == sorted(
        (K, N, 20280) for (K, N) in inputs.MXFP8_SHAPES)
    assert sorted((lin.K, lin.N, lin.M) for lin in lins["w4a16_sym"]) == sorted(
        (K, N, M) for (K, N) in inputs.W4A16_SHAPES for M in (1, 16))


def test_seeds_follow_the_recipe_and_do_not_collide():
    lins = [lin for _, lin in bench.workload_linears()] + [lin for _, lin in bench.workload_linears(True)]
    for lin in lins:
        for s in (lin.x_seed, lin.w_seed):
            assert 1000 <= s < 1100
    # within one step, no two different tensors share a seed.  Shared on purpose: one weight per
    # (K, N) for the three W4A16 row counts and for the three FP8 MLP batch sizes (X for B = 4
    # extends X for B = 1); the fused next row reuses the per-tensor linear's X and W.
    step = [lin for _, lin in bench.workload_linears()]
    x_shape, w_shape = {}, {}
    for lin in step:
        x_shape.setdefault(lin.x_seed, set()).add((lin.K, lin.x_kind, lin.x_std))
        w_shape.setdefault(lin.w_seed, set()).add((lin.N, lin.K, lin.w_std))
    assert not set(x_shape) & set(w_shape)
    # a shared seed always means the same kind of tensor (same K, or same N x K, same distribution)
    assert all(len(v) == 1 for v in x_shape.values()) and all(len(v) == 1 for v in w_shape.values())
    # so the 27 linears of a step draw 17 distinct weights: 1 + 3 (W4A16) + 2 (FP8 MLP) + 3 (MXFP8) + 8 (mixed)
    assert len(step) == 27 and len(w_shape) == 17


def test_generators_are_deterministic():
    a = inputs.outlier_channel_bf16(64, 3072, 1234)
    b = inputs.outlier_channel_bf16(64, 3072, 1234)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = inputs.normal_bf16((64, 256), 0.02, 7)
    assert torch.equal(c.view(torch.int16), inputs.normal_bf16((64, 256), 0.02, 7).view(torch.int16))
    assert not torch.equal(c.view(torch.int16), inputs.normal_bf16((64, 256), 0.02, 8).view(torch.int16))


@pytest.mark.parametrize("K,n_out", [(3072, 31), (12288, 123), (1024, 11)])
def test_outlier_channels(K, n_out):
    x, cols = inputs.outlier_channel_bf16(512, K, 1000 + K, return_cols=True)
    cols = np.asarray(cols)
    assert len(cols) == n_out == math.ceil(0.01 * K) and len(set(cols.tolist())) == n_out
    xv = x.float().numpy()
    rest = np.delete(xv, cols, axis=1)
    assert abs(rest.std() - 1.0) < 0.02 and abs(rest.mean()) < 0.01
    out = xv[:, cols]
    # 20 * t_3: heavy-tailed, scale far above the N(0,1) columns (t_3 has variance 3)
    assert np.median(np.abs(out)) > 5 * np.median(np.abs(rest))
    assert np.abs(out).max() > 100


def test_normal_generator_scale():
    w = inputs.normal_bf16((1024, 1024), 0.015, 99).float()
    assert abs(float(w.std()) - 0.015) < 0.015 * 0.01
