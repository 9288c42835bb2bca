"""The seeded workload generator: shapes, ranges, determinism (CPU)."""
import math

import numpy as np
import torch

from gated_delta_rule_43_gb300 import inputs


def test_prefill_shapes_and_ranges():
    d = inputs.make_prefill([5, 0, 7], H=3, dk=16, dv=8, dtype="bf16", seed=3, h0_sigma=0.1)
    T = 12
    assert d["q"].shape == (T, 3, 16) and d["v"].shape == (T, 3, 8)
    assert d["beta"].shape == (T, 3) and d["A_log"].shape == (3,)
    assert d["cu_seqlens"].tolist() == [0, 5, 5, 12]
    assert d["h0"].shape == (3, 3, 16, 8) and d["h0"].dtype == torch.float32
    assert d["q"].dtype == torch.bfloat16
    kn = d["k"].float().norm(dim=-1)
    assert torch.allclose(kn, torch.ones_like(kn), atol=1e-2)
    qn = d["q"].float().norm(dim=-1)
    assert torch.allclose(qn, torch.full_like(qn, 1 / math.sqrt(16)), atol=1e-2)
    b = d["beta"].float()
    assert bool((b > 0).all() and (b < 1).all())
    A = d["A_log"]
    assert bool((A >= -1).all() and (A <= 1).all())


def test_seeded_and_uniform_lengths():
    a = inputs.make_prefill(("uniform", 64, 512, 4096), H=1, dk=8, dv=8, seed=2)
    b = inputs.make_prefill(("uniform", 64, 512, 4096), H=1, dk=8, dv=8, seed=2)
    assert a["seqlens"] == b["seqlens"]
    assert all(512 <= n <= 4096 for n in a["seqlens"]) and len(a["seqlens"]) == 64
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["z"], b["z"])
    c = inputs.make_prefill(("uniform", 64, 512, 4096), H=1, dk=8, dv=8, seed=5)
    assert c["seqlens"] != a["seqlens"]


def test_host_array_bits():
    t = torch.tensor([1.0, -2.0], dtype=torch.bfloat16)
    h = inputs.host_array(t)
    assert h.dtype == np.uint16 and h.tolist() == [0x3F80, 0xC000]


def test_decode_stream():
    s = inputs.DecodeStream(4, 2, 16, 8, seed=3)
    x = s.step()
    assert x["q"].shape == (4, 2, 16) and x["v"].shape == (4, 2, 8) and x["beta"].shape == (4, 2)
    assert s.state0.shape == (4, 2, 16, 8)
    assert set(inputs.WORKLOADS) == {"tiny_fp32", "prefill_8k", "varlen_64", "decode_256",
                                     "prefill_1m", "varlen_16"}
