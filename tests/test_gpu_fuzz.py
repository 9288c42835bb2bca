"""Seeded random prefill cases against the fp64 oracle, through the C ABI.

Each case draws 1-5 packed sequences whose lengths sit on and around the tile (16) and
chunk (64) boundaries or anywhere up to 900 tokens (empty and one-token sequences
included), 1-5 heads, with or without initial states, and the default or the
long-memory gate regime.  The bf16 cases at 128/128 run the tensor-core path, the fp32
ones (head sizes 32, 64 and 128) the CUDA-core path; longer random batches (up to 3000
tokens a sequence, 8 heads) the tensor-core path again; all are scored over the whole
tensor within the stated tolerances.  Random decode batches, dense and through a state
pool, are scored the same way.
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
def test_random_long_cases_tensor_core_path(i):
    """1-6 sequences of up to 3000 tokens (many chunks each), 1-8 heads, three gate regimes."""
    rng = np.random.default_rng(70000 + i)
    n = int(rng.integers(1, 7))
    lens = [int(rng.integers(0, 3001)) for _ in range(n)]
    H = int(rng.integers(1, 9))
    h0_sigma = float(rng.choice([0.0, 0.1]))
    z_shift = float(rng.choice([0.0, -4.0, -6.0]))
    d = inputs.make_prefill(lens, H=H, dk=128, dv=128, dtype="bf16", seed=71000 + i,
                            h0_sigma=h0_sigma, z_shift=z_shift, device=DEV)
    _run_and_score(d, "bf16")


@pytest.mark.parametrize("i", range(8))
def test_random_cases_cuda_core_path(i):
    lens, H, h0_sigma, z_shift = _case(100 + i)
    dk, dv = [(32, 32), (64, 128), (128, 64), (128, 128)][i % 4]
    d = inputs.make_prefill(lens, H=H, dk=dk, dv=dv, dtype="f32", seed=3000 + i,
                            h0_sigma=h0_sigma, z_shift=z_shift, device=DEV)
    _run_and_score(d, "f32")


@pytest.mark.parametrize("i", range(8))
def test_random_decode_cases(i):
    """Random decode batches (1-40 sequences, 1-6 heads, head sizes from 32 to 128, both
    precisions, 1-5 steps), half of them through a state pool with random distinct slots:
    outputs of every step and the advanced states against the fp64 oracle."""
    import torch

    from gated_delta_rule_43_gb300 import kda
    from oracle import oracle as orc
    from tests.gpu_util import TOL, rel_l2, to_f64

    rng = np.random.default_rng(5000 + i)
    N = int(rng.integers(1, 41))
    H = int(rng.integers(1, 7))
    dk = int(rng.choice([32, 64, 128]))
    dv = int(rng.choice([32, 64, 128]))
    dtype = str(rng.choice(["f32", "bf16"]))
    steps = int(rng.integers(1, 6))
    pooled = i % 2 == 1
    ds = inputs.DecodeStream(N, H, dk, dv, dtype, seed=6000 + i, h0_sigma=0.1, device=DEV)
    A = ds.A_log.cpu().numpy().astype(np.float64)
    if pooled:
        P = N + int(rng.integers(0, 9))
        slots = torch.as_tensor(rng.permutation(P)[:N].astype(np.int32), device=DEV)
        pool = torch.zeros(P, H, dk, dv, device=DEV)
        pool.index_copy_(0, slots.long(), ds.state0)
        before = pool.clone()
    else:
        state = ds.state0.clone()
    ref_state = ds.state0.cpu().numpy().astype(np.float64)
    outs, refs = [], []
    for _ in range(steps):
        x = ds.step()
        if pooled:
            o = kda.decode_step_indexed(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log,
                                        pool, slots, check=True)
        else:
            o = kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log, state)
        h = {k: inputs.host_array(x[k]) for k in x}
        refs.append(orc.decode(h["q"], h["k"], h["v"], h["z"], h["beta"], A, ref_state))
        outs.append(to_f64(o))
    torch.cuda.synchronize()
    tol = TOL[dtype]
    got = to_f64(pool.index_select(0, slots.long())) if pooled else to_f64(state)
    assert rel_l2(np.stack(outs), np.stack(refs)) <= tol
    assert rel_l2(got, ref_state) <= tol
    if pooled:
        untouched = [s for s in range(pool.shape[0]) if s not in slots.tolist()]
        assert torch.equal(pool[untouched], before[untouched])
