"""Python side of the fp64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing in the CUDA
library or its binding imports this module.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, OpenMP over
independent (sequence, head, column-block) units); this file compiles it with
gcc and marshals numpy arrays through ctypes.  Inputs are numpy arrays in the
exact storage precision the GPU consumed: ``float64``, ``float32`` or
``uint16`` holding bf16 bit patterns.

Source of the method: "Kimi K3 Architecture: Scaling 2.8T Parameters for
Long-Context Multimodal MoE", section "The Sequence Bottleneck: Hybrid KDA and
Gated MLA" (gate equation, g_min = -5, the 16-token tile bound), with the state
update S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
o_t = S_t^T q_t.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()

G_MIN = -5.0  # lower bound of the log-decay (dev.to page, gate equation paragraph)

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile kda_oracle.c into a shared library (gcc, -O2, OpenMP, no fast-math)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P, I32, I64, D, I = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                         ctypes.c_int)
    lib.kda_oracle_gate.restype = I64
    lib.kda_oracle_gate.argtypes = [P, I, P, P, I32, I32, I32, I32, D, I, P, P]
    lib.kda_oracle_forward.restype = I
    lib.kda_oracle_forward.argtypes = [P, P, P, P, P, I, P, P, I32, I32, I32, I32, P, P, P, P, I,
                                       P, I32, D, I]
    lib.kda_oracle_decode.restype = I
    lib.kda_oracle_decode.argtypes = [P, P, P, P, P, I, P, I32, I32, I32, I32, P, P, D, I]
    lib.kda_oracle_threads.restype = I
    lib.kda_oracle_widen.restype = None
    lib.kda_oracle_widen.argtypes = [P, I, I64, P]
    return lib


def _code(a: np.ndarray) -> int:
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle input dtype {a.dtype} (want float64, float32 or uint16=bf16 bits)")


def _ptr(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """The fp64 oracle bound to one compiled library (the default, or a test variant)."""

    def __init__(self, lib_path: str | None = None):
        self._path = lib_path
        self._lib = None

    @property
    def lib(self):
        with _lock:
            if self._lib is None:
                self._lib = _bind(self._path or build())
        return self._lib

    def threads(self) -> int:
        """OpenMP threads the oracle uses by default."""
        return int(self.lib.kda_oracle_threads())

    def widen(self, a: np.ndarray) -> np.ndarray:
        """fp64 copy of an fp64 / fp32 / bf16-bits array."""
        a = np.ascontiguousarray(a)
        out = np.empty(a.shape, np.float64)
        self.lib.kda_oracle_widen(a.ctypes.data, _code(a), a.size, out.ctypes.data)
        return out

    def gate(self, z, A_log, cu_seqlens, tile: int = 16, g_min: float = G_MIN,
             softplus: bool = False):
        """g = g_min*Sigmoid(exp(A_h) z) and its in-tile inclusive cumsum.

        softplus=True evaluates the unbounded baseline g = -Softplus(exp(A_h) z)
        instead.  Returns (g, G, bad): fp64 arrays shaped like z and the number
        of tile prefix sums outside [-80, 0] or not finite.
        """
        z = np.ascontiguousarray(z)
        T, H, dk = z.shape
        A = np.ascontiguousarray(A_log, np.float64)
        cu = np.ascontiguousarray(cu_seqlens, np.int64)
        g = np.empty(z.shape, np.float64)
        G = np.empty(z.shape, np.float64)
        bad = self.lib.kda_oracle_gate(z.ctypes.data, _code(z), A.ctypes.data, cu.ctypes.data,
                                       len(cu) - 1, H, dk, tile, g_min, 1 if softplus else 0,
                                       g.ctypes.data, G.ctypes.data)
        return g, G, int(bad)

    def forward(self, q, k, v, z, beta, A_log, cu_seqlens, h0=None, *, want_o=True,
                want_state=True, o_cmp=None, col_block=None, g_min: float = G_MIN,
                nthreads: int = 0):
        """Sequential KDA recurrence over packed sequences, in fp64.

        q, k, z: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; all of one dtype
        (float64, float32, or uint16 holding bf16).  A_log: [H].  cu_seqlens:
        [N+1].  h0: [N, H, dk, dv] (any float dtype; widened to fp64) or None
        for zeros.  o_cmp: optional [T, H, dv] result (float32/float64/uint16)
        to score without materialising the fp64 output.

        Returns a dict with 'o' ([T,H,dv] fp64 or None), 'state' ([N,H,dk,dv]
        fp64 or None) and, when o_cmp is given, 'err2'/'ref2': per-(n, h) sums
        of the squared difference and of the squared reference.
        """
        q, k, v, z, beta = (np.ascontiguousarray(x) for x in (q, k, v, z, beta))
        dt = _code(q)
        for x in (k, v, z, beta):
            if _code(x) != dt:
                raise TypeError("q, k, v, z, beta must share one dtype")
        T, H, dk = q.shape
        dv = v.shape[2]
        if k.shape != (T, H, dk) or z.shape != (T, H, dk) or v.shape[:2] != (T, H) \
                or beta.shape != (T, H):
            raise ValueError("shape mismatch")
        cu = np.ascontiguousarray(cu_seqlens, np.int64)
        N = len(cu) - 1
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("bad cu_seqlens")
        A = np.ascontiguousarray(A_log, np.float64)
        h0d = None if h0 is None else np.ascontiguousarray(h0, np.float64).reshape(N, H, dk, dv)
        hT = np.empty((N, H, dk, dv), np.float64) if want_state else None
        o = np.empty((T, H, dv), np.float64) if want_o else None
        cb = col_block or (dv if N * H >= 64 else max(1, dv // 8))
        ncb = (dv + cb - 1) // cb
        err = None
        oc = None
        if o_cmp is not None:
            oc = np.ascontiguousarray(o_cmp)
            if oc.shape != (T, H, dv):
                raise ValueError("o_cmp shape")
            err = np.zeros((N, H, ncb, 2), np.float64)
        rc = self.lib.kda_oracle_forward(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, z.ctypes.data, beta.ctypes.data, dt,
            A.ctypes.data, cu.ctypes.data, N, H, dk, dv, _ptr(h0d), _ptr(hT), _ptr(o), _ptr(oc),
            0 if oc is None else _code(oc), _ptr(err), cb, g_min, nthreads)
        if rc != 0:
            raise RuntimeError("oracle rejected its arguments")
        out = {"o": o, "state": hT}
        if err is not None:
            out["err2"] = err[..., 0].sum(axis=2)
            out["ref2"] = err[..., 1].sum(axis=2)
        return out

    def decode(self, q, k, v, z, beta, A_log, state, *, g_min: float = G_MIN,
               nthreads: int = 0):
        """One decode step per sequence; `state` ([N,H,dk,dv] fp64) is updated in place.

        q, k, z: [N, H, dk]; v: [N, H, dv]; beta: [N, H].  Returns o [N, H, dv] fp64.
        """
        q, k, v, z, beta = (np.ascontiguousarray(x) for x in (q, k, v, z, beta))
        if state.dtype != np.float64 or not state.flags.c_contiguous:
            raise TypeError("state must be a C-contiguous float64 array")
        N, H, dk = q.shape
        dv = v.shape[2]
        A = np.ascontiguousarray(A_log, np.float64)
        o = np.empty((N, H, dv), np.float64)
        rc = self.lib.kda_oracle_decode(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                        z.ctypes.data, beta.ctypes.data, _code(q), A.ctypes.data,
                                        N, H, dk, dv, state.ctypes.data, o.ctypes.data, g_min,
                                        nthreads)
        if rc != 0:
            raise RuntimeError("oracle rejected its arguments")
        return o


_default = Oracle()
threads = _default.threads
widen = _default.widen
gate = _default.gate
forward = _default.forward
decode = _default.decode


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, in fp64."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = float(np.sqrt(np.sum(ref * ref)))
    num = float(np.sqrt(np.sum((x - ref) ** 2)))
    return num / den if den > 0 else num
