"""libkda.so loads on a machine without a GPU and exports exactly what include/kda.h declares.

Only host-side paths run here: version and status strings, workspace sizing,
and argument validation that returns before any CUDA call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_43_gb300 import _build, kda
    if not os.path.exists(kda.LIB_PATH):
        _build.build()
    return kda.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = header_functions()
    assert {"kda_chunk_fwd", "kda_decode_step", "kda_gate_cumsum", "kda_query_status",
            "kda_chunk_fwd_workspace_size", "kda_status_string"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in kda.h but not exported"


def test_binding_covers_the_header():
    from gated_delta_rule_43_gb300 import kda
    assert sorted(kda.SIGNATURES) == header_functions()


def test_host_only_entry_points(lib):
    from gated_delta_rule_43_gb300 import kda
    assert lib.kda_abi_version() >= 1
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert b"DECAY_RANGE" in lib.kda_status_string(kda.KDA_ERR_DECAY_RANGE)
    assert lib.kda_status_string(99) == b"KDA_ERR_UNKNOWN"
    ws = lib.kda_chunk_fwd_workspace_size(8192, 1, 32, 128, 128, kda.KDA_BF16)
    assert ws >= 256
    assert lib.kda_chunk_fwd_workspace_size(8192, 1, 32, 48, 128, kda.KDA_BF16) == 0
    assert lib.kda_decode_workspace_size() >= 16


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_argument_validation_returns_before_launch(lib):
    """Rejected arguments come back synchronously; nothing touches a device."""
    from gated_delta_rule_43_gb300 import kda
    a = 0x10000  # 256-aligned stand-in addresses; never dereferenced on these paths
    p = [_fake(a * (i + 1)) for i in range(12)]
    ws_need = lib.kda_chunk_fwd_workspace_size(64, 1, 2, 32, 32, kda.KDA_F32)

    def fwd(**kw):
        args = dict(q=p[0], k=p[1], v=p[2], z=p[3], beta=p[4], A=p[5], cu=p[6], N=1, T=64, H=2,
                    dk=32, dv=32, dt=kda.KDA_F32, h0=None, hT=None, o=p[7], ws=p[8],
                    wsb=ws_need, stream=None)
        args.update(kw)
        return lib.kda_chunk_fwd(args["q"], args["k"], args["v"], args["z"], args["beta"],
                                 args["A"], args["cu"], args["N"], args["T"], args["H"],
                                 args["dk"], args["dv"], args["dt"], args["h0"], args["hT"],
                                 args["o"], args["ws"], args["wsb"], args["stream"])

    assert fwd(dk=48) == kda.KDA_ERR_UNSUPPORTED
    assert fwd(dt=7) == kda.KDA_ERR_UNSUPPORTED
    assert fwd(q=None) == kda.KDA_ERR_INVALID_ARG
    assert fwd(cu=None) == kda.KDA_ERR_INVALID_ARG
    assert fwd(ws=None) == kda.KDA_ERR_INVALID_ARG
    assert fwd(k=_fake(a + 8)) == kda.KDA_ERR_INVALID_ARG          # misaligned
    assert fwd(ws=_fake(a * 9 + 16)) == kda.KDA_ERR_INVALID_ARG    # workspace not 256-aligned
    assert fwd(wsb=ws_need - 1) == kda.KDA_ERR_INVALID_ARG         # workspace too small
    assert fwd(o=p[0]) == kda.KDA_ERR_INVALID_ARG                  # o aliases q
    assert fwd(H=0) == kda.KDA_ERR_INVALID_ARG
    assert fwd(N=0) == kda.KDA_ERR_INVALID_ARG                     # tokens without sequences
    assert fwd(T=-1) == kda.KDA_ERR_INVALID_ARG

    def dec(**kw):
        args = dict(q=p[0], k=p[1], v=p[2], z=p[3], beta=p[4], A=p[5], S=p[6], o=p[7], N=4,
                    H=2, dk=64, dv=64, dt=kda.KDA_BF16, ws=p[8], wsb=256)
        args.update(kw)
        return lib.kda_decode_step(args["q"], args["k"], args["v"], args["z"], args["beta"],
                                   args["A"], args["S"], args["o"], args["N"], args["H"],
                                   args["dk"], args["dv"], args["dt"], args["ws"], args["wsb"],
                                   None)

    assert dec(dv=96) == kda.KDA_ERR_UNSUPPORTED
    assert dec(S=None) == kda.KDA_ERR_INVALID_ARG
    assert dec(o=p[6]) == kda.KDA_ERR_INVALID_ARG                  # o aliases the state
    assert dec(wsb=8) == kda.KDA_ERR_INVALID_ARG
    assert dec(v=_fake(a * 3 + 4)) == kda.KDA_ERR_INVALID_ARG

    def gate(**kw):
        args = dict(z=p[0], A=p[1], cu=p[2], N=1, T=64, H=2, dk=32, dt=kda.KDA_F32, C=64,
                    mode=0, G=p[3], ws=p[4], wsb=ws_need)
        args.update(kw)
        return lib.kda_gate_cumsum(args["z"], args["A"], args["cu"], args["N"], args["T"],
                                   args["H"], args["dk"], args["dt"], args["C"], args["mode"],
                                   args["G"], args["ws"], args["wsb"], None)

    assert gate(C=24) == kda.KDA_ERR_INVALID_ARG                   # not a multiple of 16
    assert gate(dk=16) == kda.KDA_ERR_UNSUPPORTED
    assert gate(G=p[0]) == kda.KDA_ERR_INVALID_ARG                 # output aliases z
    assert gate(mode=2) == kda.KDA_ERR_INVALID_ARG                 # unknown gate mode
    assert lib.kda_query_status(None, None, None) == kda.KDA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from gated_delta_rule_43_gb300 import inputs, kda
    d = inputs.make_prefill([16], H=1, dk=32, dv=32, dtype="f32")
    with pytest.raises(ValueError, match="CUDA"):
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"])
    with pytest.raises(ValueError, match="CUDA"):
        kda.decode_step(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                        torch.zeros(16, 1, 32, 32))


def test_binding_checks_shapes_and_dtypes(lib):
    """The C ABI takes raw pointers and sizes taken from q (and v): the binding refuses
    any other tensor whose shape or dtype disagrees, before anything reaches the device."""
    import torch
    from gated_delta_rule_43_gb300 import inputs, kda
    d = inputs.make_prefill([16], H=2, dk=32, dv=32, dtype="f32")
    args = [d[n] for n in ("q", "k", "v", "z", "beta", "A_log", "cu_seqlens")]

    def with_(i, t):
        a = list(args)
        a[i] = t
        return a
    with pytest.raises(TypeError, match="k has dtype"):
        kda.chunk_fwd(*with_(1, d["k"].to(torch.bfloat16)))
    with pytest.raises(ValueError, match="z has shape"):
        kda.chunk_fwd(*with_(3, d["z"][:8]))
    with pytest.raises(ValueError, match="v has shape"):
        kda.chunk_fwd(*with_(2, d["v"][:, :1].contiguous()))
    with pytest.raises(ValueError, match="beta has shape"):
        kda.chunk_fwd(*with_(4, d["beta"][:, :1].contiguous()))
    with pytest.raises(TypeError, match="A_log has dtype"):
        kda.chunk_fwd(*with_(5, d["A_log"].to(torch.bfloat16)))
    with pytest.raises(TypeError, match="cu_seqlens"):
        kda.chunk_fwd(*with_(6, d["cu_seqlens"].to(torch.int64)))
    with pytest.raises(ValueError, match="initial_state has shape"):
        kda.chunk_fwd(*args, torch.zeros(1, 2, 32, 16))
    with pytest.raises(ValueError, match="o has shape"):
        kda.chunk_fwd(*args, o=torch.empty(16, 2, 16))
    with pytest.raises(ValueError, match="final_state has shape"):
        kda.chunk_fwd_noalloc(*args, None, torch.empty(16, 2, 32), torch.empty(2, 2, 32, 32))
    with pytest.raises(ValueError, match="state has shape"):
        kda.decode_step(*args[:6], torch.zeros(16, 2, 32, 16))
    with pytest.raises(ValueError, match="state_idx has shape"):
        kda.decode_step_indexed(*args[:6], torch.zeros(20, 2, 32, 32),
                                torch.zeros(8, dtype=torch.int32))
    with pytest.raises(ValueError, match="A_log has shape"):
        kda.gate_cumsum(d["z"], d["A_log"][:1], d["cu_seqlens"])


def test_fault_hook_rejects_a_non_positive_limit(lib):
    """The bounded-wait test hook validates its limit on the host (nothing is armed)."""
    from gated_delta_rule_43_gb300 import kda
    assert lib.kda_test_chain_fault(0, 0) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_test_chain_fault(-5, -1) == kda.KDA_ERR_INVALID_ARG
