"""Thin Python binding of libkda.so (the C ABI in include/kda.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the stream.
There is no CPU fallback: if the library is missing or no GPU is present the
calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_DECAY_RANGE = 0, 1, 2, 3
KDA_ERR_TIMEOUT, KDA_ERR_CUDA, KDA_ERR_SEQLENS = 4, 5, 6
KDA_F32, KDA_BF16 = 0, 1
_DT = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}

# name -> (restype, argtypes) of every symbol include/kda.h declares
P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "kda_abi_version": (I32, []),
    "kda_status_string": (ctypes.c_char_p, [I32]),
    "kda_chunk_fwd_workspace_size": (SZ, [I64, I32, I32, I32, I32, I32]),
    "kda_chunk_fwd": (I32, [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, P, P, P, P, SZ,
                            P]),
    "kda_chunk_fwd_profiled": (I32, [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, P, P,
                                     P, P, SZ, P, ctypes.POINTER(ctypes.c_void_p), I32,
                                     ctypes.POINTER(ctypes.c_int32)]),
    "kda_chunk_fwd_segmented_workspace_size": (SZ, [I64, I32, I32, I32, I32, I32, I32]),
    "kda_chunk_fwd_segmented": (I32, [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, P, P,
                                      P, I32, P, SZ, P]),
    "kda_chunk_fwd_noalloc": (I32, [P, P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, P, P, P,
                                    P, P]),
    "kda_decode_workspace_size": (SZ, []),
    "kda_decode_step": (I32, [P, P, P, P, P, P, P, P, I32, I32, I32, I32, I32, P, SZ, P]),
    "kda_decode_step_indexed": (I32, [P, P, P, P, P, P, P, P, I32, P, I32, I32, I32, I32, I32, P,
                                      SZ, P]),
    "kda_gate_cumsum": (I32, [P, P, P, I32, I64, I32, I32, I32, I32, I32, P, P, SZ, P]),
    "kda_query_status": (I32, [P, P, ctypes.POINTER(ctypes.c_int64)]),
    "kda_test_chain_fault": (I32, [I64, I32]),
}

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str, info: int | None = None):
        self.code = code
        self.info = info
        msg = f"{where}: {status_string(code)}"
        if info is not None:
            msg += f" (info={info})"
        super().__init__(msg)


def load(path: str = LIB_PATH):
    """Load libkda.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("every tensor must live on a CUDA device (no CPU fallback)")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")


def _expect(name, t, shape, dtype=None):
    """t (when given) has exactly `shape` (and `dtype`): the C ABI takes raw pointers and
    sizes, so a tensor smaller than the sizes say would be read or written past its end."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _check_step_inputs(q, k, v, z, beta, A_log, lead):
    """q, k, z [*lead, H, dk], v [*lead, H, dv], beta [*lead, H], one dtype (fp32 or bf16);
    A_log [H] fp32.  Returns (H, dk, dv)."""
    if q.dim() != len(lead) + 2 or v.dim() != len(lead) + 2:
        raise ValueError(f"q and v must be [{', '.join(map(str, lead))}, H, D]")
    H, dk = q.shape[-2:]
    dv = v.shape[-1]
    if q.dtype not in _DT:
        raise TypeError(f"q has dtype {q.dtype}; fp32 and bf16 are supported")
    _expect("k", k, (*lead, H, dk), q.dtype)
    _expect("z", z, (*lead, H, dk), q.dtype)
    _expect("v", v, (*lead, H, dv), q.dtype)
    _expect("beta", beta, (*lead, H), q.dtype)
    _expect("A_log", A_log, (H,), torch.float32)
    return H, dk, dv


def _check_prefill(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state):
    if q.dim() != 3:
        raise ValueError("q must be [T, H, dk]")
    T = q.shape[0]
    H, dk, dv = _check_step_inputs(q, k, v, z, beta, A_log, (T,))
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1 or cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be a 1-D int32 tensor [N + 1]")
    N = cu_seqlens.numel() - 1
    _expect("initial_state", initial_state, (N, H, dk, dv), torch.float32)
    _expect("final_state", final_state, (N, H, dk, dv), torch.float32)
    _expect("o", o, (T, H, dv), q.dtype)
    return T, N, H, dk, dv


def chunk_fwd_workspace_size(total_tokens: int, num_seqs: int, H: int, dk: int, dv: int,
                             dtype: torch.dtype) -> int:
    return int(load().kda_chunk_fwd_workspace_size(total_tokens, num_seqs, H, dk, dv,
                                                   _DT[dtype]))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def chunk_fwd(q, k, v, z, beta, A_log, cu_seqlens, initial_state=None, *,
              output_final_state: bool = True, o=None, final_state=None, workspace=None,
              stream=None, check: bool = False):
    """KDA chunked prefill over packed sequences (kda_chunk_fwd).

    q, k, z [T, H, dk], v [T, H, dv], beta [T, H] (fp32 or bf16, one dtype);
    A_log [H] fp32; cu_seqlens [N+1] int32; initial_state [N, H, dk, dv] fp32
    or None.  Returns (o [T, H, dv], final_state [N, H, dk, dv] fp32 or None).
    ``final_state`` may be passed as ``initial_state`` for an in-place update.
    With ``check=True`` the stream is synchronised and a device-side error
    raises KdaError.
    """
    lib = load()
    T, N, H, dk, dv = _check_prefill(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o,
                                     final_state)
    _check_cuda(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state, workspace)
    dt = _DT[q.dtype]
    if o is None:
        o = torch.empty(T, H, dv, dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    need = int(lib.kda_chunk_fwd_workspace_size(T, N, H, dk, dv, dt))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    rc = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A_log),
                           _ptr(cu_seqlens), N, T, H, dk, dv, dt, _ptr(initial_state),
                           _ptr(final_state), _ptr(o), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd")
    if check:
        query_status(workspace, stream, raise_on_error=True)
    return o, final_state


def chunk_fwd_segmented(q, k, v, z, beta, A_log, cu_seqlens, initial_state=None, *,
                        segments: int, output_final_state: bool = True, o=None,
                        final_state=None, workspace=None, stream=None, check: bool = False):
    """Segment-parallel prefill (kda_chunk_fwd_segmented): chunk_fwd's arguments and
    results, each sequence's chunks of a window cut into up to ``segments`` segments."""
    lib = load()
    T, N, H, dk, dv = _check_prefill(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o,
                                     final_state)
    _check_cuda(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state, workspace)
    dt = _DT[q.dtype]
    if o is None:
        o = torch.empty(T, H, dv, dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    need = int(lib.kda_chunk_fwd_segmented_workspace_size(T, N, H, dk, dv, dt, int(segments)))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    rc = lib.kda_chunk_fwd_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta),
                                     _ptr(A_log), _ptr(cu_seqlens), N, T, H, dk, dv, dt,
                                     _ptr(initial_state), _ptr(final_state), _ptr(o),
                                     int(segments), _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_segmented")
    if check:
        query_status(workspace, stream, raise_on_error=True)
    return o, final_state


def chunk_fwd_profiled(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state,
                       workspace, events, stream=None) -> int:
    """kda_chunk_fwd with CUDA events recorded around each kernel it launches.

    `events` is a list of torch.cuda.Event(enable_timing=True); returns how many
    were recorded.  Kernel j of the call runs between events[2j] and events[2j+1],
    both recorded on the stream that kernel was launched on.
    """
    lib = load()
    T, N, H, dk, dv = _check_prefill(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o,
                                     final_state)
    _check_cuda(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state, workspace)
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record(stream if stream is not None else torch.cuda.current_stream())
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    used = ctypes.c_int32(0)
    rc = lib.kda_chunk_fwd_profiled(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A_log),
                                    _ptr(cu_seqlens), N, T, H, dk, dv, _DT[q.dtype],
                                    _ptr(initial_state), _ptr(final_state), _ptr(o),
                                    _ptr(workspace), workspace.numel(), _stream(stream),
                                    handles, len(events), ctypes.byref(used))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_profiled")
    return used.value


def chunk_fwd_noalloc(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state,
                      status_out=None, stream=None):
    """kda_chunk_fwd_noalloc: the chunked forward with the library's own fixed scratch.

    For callers that cannot allocate device memory; o, final_state and the
    optional 16-byte status_out buffer are supplied by the caller.  Work on the
    shared scratch must not overlap between calls (serialise them).
    """
    lib = load()
    T, N, H, dk, dv = _check_prefill(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o,
                                     final_state)
    _check_cuda(q, k, v, z, beta, A_log, cu_seqlens, initial_state, o, final_state, status_out)
    if status_out is not None and status_out.numel() * status_out.element_size() < 16:
        raise ValueError("status_out must hold at least 16 bytes")
    rc = lib.kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A_log),
                                   _ptr(cu_seqlens), N, T, H, dk, dv, _DT[q.dtype],
                                   _ptr(initial_state), _ptr(final_state), _ptr(o),
                                   _ptr(status_out), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_noalloc")
    return o, final_state


def decode_step(q, k, v, z, beta, A_log, state, *, o=None, workspace=None, stream=None):
    """One decode step for N sequences (kda_decode_step); `state` is updated in place.

    q, k, z [N, H, dk], v [N, H, dv], beta [N, H]; state [N, H, dk, dv] fp32.
    Returns o [N, H, dv].
    """
    lib = load()
    if q.dim() != 3:
        raise ValueError("q must be [N, H, dk]")
    N = q.shape[0]
    H, dk, dv = _check_step_inputs(q, k, v, z, beta, A_log, (N,))
    _expect("state", state, (N, H, dk, dv), torch.float32)
    _expect("o", o, (N, H, dv), q.dtype)
    _check_cuda(q, k, v, z, beta, A_log, state, o, workspace)
    if o is None:
        o = torch.empty(N, H, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(int(lib.kda_decode_workspace_size()), q.device)
    rc = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A_log),
                             _ptr(state), _ptr(o), N, H, dk, dv, _DT[q.dtype], _ptr(workspace),
                             workspace.numel(), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")
    return o


def decode_step_indexed(q, k, v, z, beta, A_log, state_pool, state_idx, *, o=None,
                        workspace=None, stream=None, check: bool = False):
    """One decode step where sequence n owns slot state_idx[n] of state_pool (in place).

    q, k, z [N, H, dk], v [N, H, dv], beta [N, H]; state_pool [P, H, dk, dv] fp32;
    state_idx [N] int32 (distinct values in [0, P)).  Returns o [N, H, dv].
    """
    lib = load()
    if q.dim() != 3 or state_pool.dim() != 4:
        raise ValueError("q must be [N, H, dk] and state_pool [P, H, dk, dv]")
    N = q.shape[0]
    H, dk, dv = _check_step_inputs(q, k, v, z, beta, A_log, (N,))
    _expect("state_pool", state_pool, (state_pool.shape[0], H, dk, dv), torch.float32)
    _expect("state_idx", state_idx, (N,), torch.int32)
    _expect("o", o, (N, H, dv), q.dtype)
    _check_cuda(q, k, v, z, beta, A_log, state_pool, state_idx, o, workspace)
    if o is None:
        o = torch.empty(N, H, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(int(lib.kda_decode_workspace_size()), q.device)
    rc = lib.kda_decode_step_indexed(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta),
                                     _ptr(A_log), _ptr(state_pool), _ptr(state_idx),
                                     state_pool.shape[0], _ptr(o), N, H, dk, dv, _DT[q.dtype],
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step_indexed")
    if check:
        query_status(workspace, stream, raise_on_error=True)
    return o


def gate_cumsum(z, A_log, cu_seqlens, chunk: int = 64, *, softplus: bool = False,
                workspace=None, stream=None, check: bool = False):
    """The standalone gate kernel (kda_gate_cumsum): fp32 in-chunk cumsum of g [T, H, dk].

    softplus=True evaluates the unbounded -Softplus baseline instead of the
    lower-bounded gate (same 16-token range check)."""
    lib = load()
    if z.dim() != 3 or z.dtype not in _DT:
        raise ValueError("z must be [T, H, dk], fp32 or bf16")
    T, H, dk = z.shape
    _expect("A_log", A_log, (H,), torch.float32)
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1 or cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be a 1-D int32 tensor [N + 1]")
    _check_cuda(z, A_log, cu_seqlens, workspace)
    N = cu_seqlens.numel() - 1
    G = torch.empty(T, H, dk, dtype=torch.float32, device=z.device)
    dt = _DT[z.dtype]
    if workspace is None:
        workspace = alloc_workspace(int(lib.kda_chunk_fwd_workspace_size(T, N, H, dk, dk, dt)),
                                    z.device)
    rc = lib.kda_gate_cumsum(_ptr(z), _ptr(A_log), _ptr(cu_seqlens), N, T, H, dk, dt, chunk,
                             1 if softplus else 0, _ptr(G), _ptr(workspace), workspace.numel(),
                             _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_gate_cumsum")
    if check:
        query_status(workspace, stream, raise_on_error=True)
    return G, workspace


def query_status(workspace, stream=None, *, raise_on_error: bool = False):
    """(code, info) recorded in `workspace` by the last call (synchronises the stream)."""
    info = ctypes.c_int64(0)
    rc = load().kda_query_status(_ptr(workspace), _stream(stream), ctypes.byref(info))
    if raise_on_error and rc != KDA_OK:
        raise KdaError(rc, "device status", info.value)
    return rc, info.value
