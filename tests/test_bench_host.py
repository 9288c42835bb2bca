"""Host logic of bench.py: the roofline conventions and the multi-rank reduction (CPU, gloo)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_algorithmic_conventions():
    # 1282 bytes per token-head at dk = dv = 128 in bf16 (q, k, z, v, beta in; o out)
    assert bench.prefill_bytes([1], 1, 128, 128, 2, False, False) == 1282
    # plus 64 KiB of fp32 state per (sequence, head) in or out
    assert bench.prefill_bytes([8192], 32, 128, 128, 2, False, True) == \
        8192 * 32 * 1282 + 32 * 128 * 128 * 4
    # 139,264 flops per token-head under the fixed convention
    assert bench.prefill_flops([1], 1, 128, 128) == 139264


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r "took" 1 + r seconds for 100 units: weak scaling divides world*units by the max
    thr, tmax = bench.aggregate(100.0, 1.0 + rank, world)
    out[rank] = (thr, tmax)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_weak_scaling_reduction_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    for r in range(2):
        thr, tmax = out[r]
        assert tmax == 2.0 and thr == pytest.approx(100.0 * 2 / 2.0)


def test_single_rank_reduction_is_identity():
    assert bench.aggregate(50.0, 2.0, 1) == (25.0, 2.0)


class _FakeCudart:
    """Stands in for torch.cuda.cudart() on a machine without a GPU: records the
    registrations and answers with the given status."""

    def __init__(self, status=0):
        self.status = status
        self.registered = {}

    def cudaHostRegister(self, ptr, size, flags):
        if self.status == 0:
            self.registered[ptr] = size
        return self.status

    def cudaHostUnregister(self, ptr):
        self.registered.pop(ptr)
        return 0


def test_host_buffers_are_huge_page_mappings_registered_and_released(monkeypatch):
    """bench.HostBuffers: each tensor lives in a mapping rounded up to 2 MiB, registered
    whole with the driver, viewed with the asked shape and dtype; release() unregisters
    every mapping."""
    import torch
    fake = _FakeCudart()
    monkeypatch.setattr(torch.cuda, "cudart", lambda: fake)
    hb = bench.HostBuffers()
    a = hb.new((3, 5, 7), torch.bfloat16)
    b = hb.new((1000, 700), torch.float32)
    assert a.shape == (3, 5, 7) and a.dtype == torch.bfloat16
    assert b.shape == (1000, 700) and b.dtype == torch.float32
    assert hb.kind == "huge-page registered"
    assert sorted(fake.registered.values()) == [2 << 20, 4 << 20]   # 2,800,000 B -> 4 MiB
    b.fill_(1.5)
    a.fill_(-2.0)
    assert float(b.sum()) == 1.5 * 700000 and float(a[2, 4, 6]) == -2.0
    hb.release()
    assert fake.registered == {}


def test_host_buffers_fall_back_to_pinned_when_registration_fails(monkeypatch):
    import torch
    monkeypatch.setattr(torch.cuda, "cudart", lambda: _FakeCudart(status=1))
    calls = []
    real_empty = torch.empty

    def fake_empty(*shape, **kw):
        if kw.pop("pin_memory", False):
            calls.append(shape)
        return real_empty(*shape, **kw)
    monkeypatch.setattr(torch, "empty", fake_empty)
    hb = bench.HostBuffers()
    t = hb.new((4, 4), torch.float32)
    assert t.shape == (4, 4) and hb.kind == "pinned" and calls == [((4, 4),)]
