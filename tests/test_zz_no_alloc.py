"""kda_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate device memory.

A caller that is handed only its input and output buffers (a plug-in inside an
application that owns every device allocation, or a serving loop that must not
call cudaMalloc after start-up) cannot supply kda_chunk_fwd's workspace; this
entry point takes its scratch from a fixed array inside the library instead.

The test calls it through the C ABI twice in a row on different problems (so the
second call runs on top of the first call's leftovers in the shared array) and
compares each result with kda_chunk_fwd's within the parity tolerance, checks
the status word it copies out, and checks that a problem too large for the
array is refused before anything is launched.  The file is named to be
collected last.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from tests.gpu_util import TOL, rel_l2, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(d, o, hT, status):
    """kda_chunk_fwd_noalloc through the C ABI (argument marshalling only)."""
    lib = kda.load()
    T, H, dk = d["q"].shape
    dv = d["v"].shape[-1]
    N = d["cu_seqlens"].numel() - 1
    dt = kda.KDA_BF16 if d["q"].dtype == torch.bfloat16 else kda.KDA_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kda_chunk_fwd_noalloc(_p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["z"]),
                                     _p(d["beta"]), _p(d["A_log"]), _p(d["cu_seqlens"]), N, T,
                                     H, dk, dv, dt, _p(d["h0"]), _p(hT), _p(o), _p(status),
                                     stream)


def _check_against_workspace_entry(d, dtype):
    T, H, _ = d["q"].shape
    N = d["cu_seqlens"].numel() - 1
    dv = d["v"].shape[-1]
    dk = d["q"].shape[-1]
    o = torch.full((T, H, dv), float("nan"), dtype=d["q"].dtype, device=DEV)
    hT = torch.full((N, H, dk, dv), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.full((16,), 0xFF, dtype=torch.uint8, device=DEV)
    rc = _call_noalloc(d, o, hT, status)
    assert rc == kda.KDA_OK, kda.status_string(rc)
    code, info = kda.query_status(status)
    assert code == kda.KDA_OK, (kda.status_string(code), info)
    o_ref, s_ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                                 d["cu_seqlens"], d["h0"], check=True)
    tol = TOL[dtype]
    e_o = rel_l2(to_f64(o), to_f64(o_ref))
    e_s = rel_l2(to_f64(hT), to_f64(s_ref))
    assert e_o <= tol and e_s <= tol, (e_o, e_s)


def test_two_calls_in_a_row_match_the_workspace_entry():
    # first call: tensor-core path, packed sequences with an empty one, initial state
    d1 = inputs.make_prefill([700, 0, 1500], H=4, dk=128, dv=128, dtype="bf16", seed=41,
                             h0_sigma=0.1, device=DEV)
    _check_against_workspace_entry(d1, "bf16")
    # second call, right after: a longer sequence that needs several windows of the
    # fixed scratch (more heads, fewer records fit), no initial state
    # (8 heads: 56 chunk slots of records fit the array, the sequence has 79)
    d2 = inputs.make_prefill([5000], H=8, dk=128, dv=128, dtype="bf16", seed=42, device=DEV)
    _check_against_workspace_entry(d2, "bf16")


def test_running_state_in_the_scratch_across_windows():
    """Tensor-core path with final_state NULL: the running state lives in the library's
    array beside the chunk records, and the sequence is long enough that its chunks run
    in several windows of records, so the state crosses windows inside the array.  o
    matches kda_chunk_fwd's."""
    d = inputs.make_prefill([20000, 333], H=4, dk=128, dv=128, dtype="bf16", seed=44,
                            h0_sigma=0.1, z_shift=-4.0, device=DEV)
    T, H, dv = d["v"].shape
    o = torch.full((T, H, dv), float("nan"), dtype=torch.bfloat16, device=DEV)
    status = torch.full((16,), 0xFF, dtype=torch.uint8, device=DEV)
    rc = _call_noalloc(d, o, None, status)
    assert rc == kda.KDA_OK, kda.status_string(rc)
    code, info = kda.query_status(status)
    assert code == kda.KDA_OK, (kda.status_string(code), info)
    o_ref, _ = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                             d["cu_seqlens"], d["h0"], output_final_state=False, check=True)
    assert rel_l2(to_f64(o), to_f64(o_ref)) <= TOL["bf16"]


def test_cuda_core_path_in_place():
    d = inputs.make_prefill([90, 33], H=2, dk=64, dv=32, dtype="f32", seed=43, h0_sigma=0.1,
                            device=DEV)
    _check_against_workspace_entry(d, "f32")


def test_too_large_is_refused_before_launch():
    lib = kda.load()
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(10)]
    # one record per head (74,240 bytes) no longer fits 32 MiB at H = 500
    rc = lib.kda_chunk_fwd_noalloc(*fake[:7], 1, 64, 500, 128, 128, kda.KDA_BF16, None,
                                   fake[7], fake[8], None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    # the running state of 64 x 32 heads (128 MiB) does not fit when final_state is NULL
    rc = lib.kda_chunk_fwd_noalloc(*fake[:7], 64, 64 * 64, 32, 128, 128, kda.KDA_BF16, None,
                                   None, fake[8], None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
