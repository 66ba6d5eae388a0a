"""The seeded input generator against its stated recipe: the workload table,
the value distributions, reproducibility and the draw order.  Every parity
test and the bench draw their operands here, so a drift in it would change
what every other test checks."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import gemm_inputs

# The recipe: name -> (M, N, K, dtype, distribution, seed)
RECIPE = {
    "gemm_256_f16": (256, 256, 256, "f16", "uniform", 0),
    "gemm_256_f16_int": (256, 256, 256, "f16", "int", 0),
    "gemm_4096_f16": (4096, 4096, 4096, "f16", "normal_scaled", 1),
    "gemm_8192_f16": (8192, 8192, 8192, "f16", "normal_scaled", 2),
    "gelu_3072x16384x4096_bf16": (3072, 16384, 4096, "bf16", "normal_xw", 3),
    "ragged_4095x4097x8191_f16": (4095, 4097, 8191, "f16", "uniform", 4),
    "skinny_64x8192x8192_f16": (64, 8192, 8192, "f16", "uniform", 4),
    "mosaic_16896x512x640_f16": (16896, 512, 640, "f16", "uniform01", 42),
}


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().copy()


def test_workload_table_is_the_recipe():
    assert set(gemm_inputs.WORKLOADS) == set(RECIPE)
    for name, (M, N, K, dt, dist, seed) in RECIPE.items():
        w = gemm_inputs.WORKLOADS[name]
        assert (w.M, w.N, w.K, w.dtype, w.dist, w.seed) == (M, N, K, dt, dist, seed), name
        assert w.epilogue == ("gelu" if name.startswith("gelu") else "none")
        assert w.flops == 2 * M * N * K


@pytest.mark.parametrize("name", sorted(RECIPE))
def test_distribution_of_each_workload(name):
    w = gemm_inputs.WORKLOADS[name]
    # a reduced draw of the same recipe (K kept where it sets the scale)
    A, B = gemm_inputs.make(w, M=96, N=80, K=w.K if w.dist == "normal_scaled" else 512)
    td = torch.float16 if w.dtype == "f16" else torch.bfloat16
    assert A.dtype == td and B.dtype == td and A.shape[0] == 96 and B.shape[0] == 80
    a, b = A.double().numpy(), B.double().numpy()
    if w.dist == "uniform":
        for x in (a, b):
            assert x.min() >= -1 and x.max() <= 1 and abs(x.mean()) < 0.02
            assert abs(x.std() - 1 / math.sqrt(3)) < 0.01        # U[-1,1]: sd 1/sqrt(3)
    elif w.dist == "uniform01":
        for x in (a, b):
            assert x.min() >= 0 and x.max() <= 1 and abs(x.mean() - 0.5) < 0.01
    elif w.dist == "normal_scaled":
        for x in (a, b):
            assert abs(x.std() * math.sqrt(w.K) - 1) < 0.03 and abs(x.mean()) * math.sqrt(w.K) < 0.03
    elif w.dist == "normal_xw":
        assert abs(a.std() - 1) < 0.02                            # X ~ N(0, 1)
        assert abs(b.std() / 0.02 - 1) < 0.02                     # W ~ N(0, 0.02)
    elif w.dist == "int":
        for x in (a, b):
            assert set(np.unique(x)) <= {-2.0, -1.0, 0.0, 1.0, 2.0} and np.all(x == np.round(x))
    else:
        raise AssertionError(w.dist)


def test_draws_are_reproducible_and_seeded():
    a1, b1 = gemm_inputs.make("gemm_256_f16")
    a2, b2 = gemm_inputs.make("gemm_256_f16")
    assert np.array_equal(_bits(a1), _bits(a2)) and np.array_equal(_bits(b1), _bits(b2))
    a3, _ = gemm_inputs.make("gemm_256_f16", seed=1)
    assert not np.array_equal(_bits(a1), _bits(a3))
    assert not np.array_equal(_bits(a1), _bits(b1))             # A and B are separate draws


def test_a_is_drawn_before_b_and_cast_to_nearest_even():
    w = gemm_inputs.WORKLOADS["gemm_256_f16"]
    g = torch.Generator().manual_seed(w.seed)
    a = torch.rand((w.M, w.K), generator=g) * 2 - 1
    b = torch.rand((w.N, w.K), generator=g) * 2 - 1
    A, B = gemm_inputs.make(w)
    assert np.array_equal(_bits(A), _bits(a.half())) and np.array_equal(_bits(B), _bits(b.half()))


def test_integer_copy_is_the_second_draw_of_seed_0():
    w = gemm_inputs.WORKLOADS["gemm_256_f16_int"]
    g = torch.Generator().manual_seed(0)
    torch.rand((256, 256), generator=g)                          # the float pair first
    torch.rand((256, 256), generator=g)
    a = torch.randint(-2, 3, (256, 256), generator=g).float()
    b = torch.randint(-2, 3, (256, 256), generator=g).float()
    A, B = gemm_inputs.make(w)
    assert np.array_equal(_bits(A), _bits(a.half())) and np.array_equal(_bits(B), _bits(b.half()))


def test_custom_shapes_and_bias():
    A, B = gemm_inputs.custom(33, 17, 70, dtype="bf16", dist="int", seed=5, lo=-3, hi=3)
    assert A.shape == (33, 70) and B.shape == (17, 70) and A.dtype == torch.bfloat16
    assert A.double().abs().max() <= 3
    bi = gemm_inputs.bias(1000, "f16", seed=5, dist="int", lo=-4, hi=4)
    assert bi.shape == (1000,) and set(np.unique(bi.double().numpy())) <= set(range(-4, 5))
    bu = gemm_inputs.bias(1000, "bf16", seed=5)
    assert bu.dtype == torch.bfloat16 and bu.double().min() >= -0.5 and bu.double().max() <= 0.5
    # the bias has a generator of its own: were it drawn from the operands'
    # stream of the same seed, it would be exactly half of A's first row
    # (U[-0.5, 0.5] against U[-1, 1] from the same uniforms; x2 is exact)
    a, _ = gemm_inputs.custom(1, 1, 1000, dtype="bf16", seed=5)
    assert a.shape == (1, 1000)
    assert not torch.equal(bu * 2, a.reshape(-1))
