"""Seeded random prefill cases against the fp64 oracle, through the C ABI.

Each case draws 1-5 packed sequences whose lengths sit on and around the tile (16) and
chunk (64) boundaries or anywhere up to 900 tokens (empty and one-token sequences
included), 1-5 heads, with or without initial states, and the default or the
long-memory gate regime.  The bf16 cases at 128/128 run the tensor-core path, the fp32
ones (head sizes 32, 64 and 128) the CUDA-core path; all are scored over the whole
tensor within the stated tolerances.
"""
import numpy as np
import pytest

from gated_delta_rule_43_gb300 import inputs
from tests.test_gpu_prefill import _run_and_score

pytestmark = pytest.mark.gpu
DEV = "cuda"
EDGES = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 191, 300, 777]


def _case(i: int):
    rng = np.random.default_rng(1000 + i)
    n = int(rng.integers(1, 6))
    lens = [int(rng.choice(EDGES)) if rng.random() < 0.6 else int(rng.integers(0, 900))
            for _ in range(n)]
    H = int(rng.integers(1, 6))
    h0_sigma = float(rng.choice([0.0, 0.1]))
    z_shift = float(rng.choice([0.0, -4.0]))
    return lens, H, h0_sigma, z_shift


@pytest.mark.parametrize("i", range(16))
def test_random_cases_tensor_core_path(i):
    lens, H, h0_sigma, z_shift = _case(i)
    d = inputs.make_prefill(lens, H=H, dk=128, dv=128, dtype="bf16", seed=2000 + i,
                            h0_sigma=h0_sigma, z_shift=z_shift, device=DEV)
    _run_and_score(d, "bf16")


@pytest.mark.parametrize("i", range(8))
def test_random_cases_cuda_core_path(i):
    lens, H, h0_sigma, z_shift = _case(100 + i)
    dk, dv = [(32, 32), (64, 128), (128, 64), (128, 128)][i % 4]
    d = inputs.make_prefill(lens, H=H, dk=dk, dv=dv, dtype="f32", seed=3000 + i,
                            h0_sigma=h0_sigma, z_shift=z_shift, device=DEV)
    _run_and_score(d, "f32")
