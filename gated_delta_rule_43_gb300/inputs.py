"""Seeded synthetic inputs for KDA workloads (shared by the tests, smoke check and bench).

This module only draws random numbers and arranges them; it holds none of the
method's arithmetic (no gate, no recurrence).  The distributions follow the
workload recipe used throughout this project: q, k ~ N(0, 1) then L2-normalised
per (token, head) over dk, q scaled by 1/sqrt(dk); v ~ N(0, 1); z ~ N(0, 1) per
channel; A ~ U(-1, 1) per head; beta = Sigmoid(N(0, 1)) (beta is an input of the
method, supplied already squashed into (0, 1)); optional initial state
~ N(0, sigma^2) in fp32.  Normalisation is done in fp32 before rounding to the
storage dtype.

Draw order (fixed, one torch.Generator per workload): sequence lengths (if
random), q, k, v, z, A, beta-pre, initial state; decode draws A and the state
first and then, per step, q, k, v, z, beta-pre.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One synthetic KDA workload.

    kind      "prefill" (packed sequences through the chunked forward) or
              "decode" (N sequences, one token per step, resident state).
    seqlens   prefill: a tuple of lengths, or ("uniform", count, lo, hi)
              for integer lengths drawn uniformly from [lo, hi] inclusive.
    """
    name: str
    kind: str
    H: int
    dk: int
    dv: int
    dtype: str
    seed: int
    seqlens: tuple = ()
    h0_sigma: float = 0.0
    N: int = 0
    steps: int = 0
    chunk: int = 0
    notes: str = field(default="", compare=False)


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", "prefill", H=2, dk=32, dv=32, dtype="f32", seed=0, seqlens=(64,),
        chunk=16, notes="B=1, T=64, fp32, chunk 16, zero initial state"),
    "prefill_8k": Workload(
        "prefill_8k", "prefill", H=32, dk=128, dv=128, dtype="bf16", seed=1, seqlens=(8192,),
        notes="B=1, T=8192, bf16, zero initial state, emits the fp32 final state"),
    "varlen_64": Workload(
        "varlen_64", "prefill", H=32, dk=128, dv=128, dtype="bf16", seed=2,
        seqlens=("uniform", 64, 512, 4096), h0_sigma=0.1,
        notes="64 packed sequences, lengths U[512, 4096], initial state N(0, 0.01)"),
    "decode_256": Workload(
        "decode_256", "decode", H=32, dk=128, dv=128, dtype="bf16", seed=3, N=256, steps=128,
        h0_sigma=0.1, notes="256 sequences x 1 token, fp32 state N(0, 0.01) in place"),
    "prefill_1m": Workload(
        "prefill_1m", "prefill", H=16, dk=128, dv=128, dtype="bf16", seed=4,
        seqlens=(1048576,), notes="B=1, T=1,048,576, bf16, carried state, final state"),
    # a smaller packed case of the varlen recipe, for kernel profiles that must hold only a
    # few GB on the device (the 128-column chain kernel runs on it as on varlen_64)
    "varlen_16": Workload(
        "varlen_16", "prefill", H=32, dk=128, dv=128, dtype="bf16", seed=5,
        seqlens=("uniform", 16, 512, 4096), h0_sigma=0.1,
        notes="16 packed sequences, lengths U[512, 4096], initial state N(0, 0.01)"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_seqlens(spec, gen: torch.Generator) -> list[int]:
    if len(spec) == 4 and spec[0] == "uniform":
        _, count, lo, hi = spec
        return torch.randint(lo, hi + 1, (count,), generator=gen,
                             device=gen.device).cpu().tolist()
    return [int(x) for x in spec]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    # input preparation: unit L2 norm over the last axis, in fp32
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def make_prefill(seqlens, H: int, dk: int, dv: int, dtype: str = "bf16", *, seed: int = 0,
                 h0_sigma: float = 0.0, z_shift: float = 0.0, device="cpu",
                 gen: torch.Generator | None = None):
    """Packed prefill inputs.  Returns a dict of tensors on `device`:

    q, k, z [T, H, dk] and v [T, H, dv] in `dtype`; beta [T, H] in `dtype`;
    A_log [H] fp32; cu_seqlens [N+1] int32; h0 [N, H, dk, dv] fp32 or None.
    `seqlens` may be a list of lengths or a ("uniform", count, lo, hi) spec.
    z ~ N(z_shift, 1): the default centres the gate near g = -2.5 (the state keeps a
    token for about one step); z_shift = -4 gives g near -0.05 per token, a memory of
    tens to hundreds of tokens, across many chunks.
    """
    gen = gen or _gen(seed, device)
    lens = draw_seqlens(tuple(seqlens), gen)
    T = int(sum(lens))
    N = len(lens)
    td = DTYPES[dtype]
    f32 = dict(device=device, dtype=torch.float32, generator=gen)
    q = _unit_rows(torch.randn(T, H, dk, **f32)) * (1.0 / math.sqrt(dk))
    k = _unit_rows(torch.randn(T, H, dk, **f32))
    v = torch.randn(T, H, dv, **f32)
    z = torch.randn(T, H, dk, **f32) + z_shift
    A = torch.rand(H, **f32) * 2.0 - 1.0
    beta = torch.sigmoid(torch.randn(T, H, **f32))
    h0 = torch.randn(N, H, dk, dv, **f32) * h0_sigma if h0_sigma > 0 else None
    cu = torch.zeros(N + 1, dtype=torch.int32, device=device)
    if N:
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64, device=device), 0).to(
            torch.int32)
    return {"q": q.to(td), "k": k.to(td), "v": v.to(td), "z": z.to(td), "beta": beta.to(td),
            "A_log": A, "cu_seqlens": cu, "h0": h0, "seqlens": lens}


def make_workload(w: Workload, device="cpu"):
    """Inputs of a prefill workload (see WORKLOADS)."""
    if w.kind != "prefill":
        raise ValueError("make_workload is for prefill workloads; use DecodeStream")
    return make_prefill(w.seqlens, w.H, w.dk, w.dv, w.dtype, seed=w.seed, h0_sigma=w.h0_sigma,
                        device=device)


class DecodeStream:
    """Seeded decode inputs: the initial state, then fresh per-step token inputs."""

    def __init__(self, N: int, H: int, dk: int, dv: int, dtype: str = "bf16", *, seed: int = 0,
                 h0_sigma: float = 0.1, device="cpu"):
        self.N, self.H, self.dk, self.dv = N, H, dk, dv
        self.td = DTYPES[dtype]
        self.gen = _gen(seed, device)
        self.device = device
        f32 = dict(device=device, dtype=torch.float32, generator=self.gen)
        self.A_log = torch.rand(H, **f32) * 2.0 - 1.0
        self.state0 = torch.randn(N, H, dk, dv, **f32) * h0_sigma

    def step(self):
        """Inputs of one decode step: q, k, z [N, H, dk], v [N, H, dv], beta [N, H]."""
        N, H, dk, dv = self.N, self.H, self.dk, self.dv
        f32 = dict(device=self.device, dtype=torch.float32, generator=self.gen)
        q = _unit_rows(torch.randn(N, H, dk, **f32)) * (1.0 / math.sqrt(dk))
        k = _unit_rows(torch.randn(N, H, dk, **f32))
        v = torch.randn(N, H, dv, **f32)
        z = torch.randn(N, H, dk, **f32)
        beta = torch.sigmoid(torch.randn(N, H, **f32))
        td = self.td
        return {"q": q.to(td), "k": k.to(td), "v": v.to(td), "z": z.to(td), "beta": beta.to(td)}


def decode_workload(w: Workload, device="cpu") -> DecodeStream:
    return DecodeStream(w.N, w.H, w.dk, w.dv, w.dtype, seed=w.seed, h0_sigma=w.h0_sigma,
                        device=device)


def host_array(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor in its exact storage precision (bf16 -> uint16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
