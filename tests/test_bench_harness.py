"""The benchmark harness on the CPU: its timing helpers run with CUDA replaced by stand-ins, and the
readout measurement rotates buffer sets that span at least three times the L2 cache, so its HBM
figure cannot come from L2."""
import contextlib
import types

import torch

import bench


class _Event:
    def __init__(self, enable_timing=False):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return 1.0


class _Stream:
    cuda_stream = 0

    def wait_stream(self, other):
        pass


class _Graph:
    def replay(self):
        pass


def _fake_cuda(monkeypatch, l2_bytes):
    monkeypatch.setattr(torch.cuda, "Event", _Event)
    monkeypatch.setattr(torch.cuda, "Stream", lambda *a, **k: _Stream())
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a, **k: _Stream())
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    monkeypatch.setattr(torch.cuda, "graph", lambda g, **k: contextlib.nullcontext())
    monkeypatch.setattr(torch.cuda, "CUDAGraph", _Graph)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda d: types.SimpleNamespace(L2_cache_size=l2_bytes))


def test_readout_rotation_spans_three_l2(monkeypatch):
    l2 = 126 * 1024 * 1024
    _fake_cuda(monkeypatch, l2)
    calls = []
    lib = types.SimpleNamespace(readout_decide=lambda *a: calls.append(a[7].data_ptr()))  # the set's p_cal
    ms, nbytes, gms, one, (n_sets, rot_bytes) = bench.measure_readout(lib, torch, torch.device("cpu"), _Stream(),
                                                                      reps=8, timing_forms=True)
    assert rot_bytes >= 3 * l2 and n_sets >= 2
    assert nbytes == 7080112            # 65,536 questions: 2 n 4 + 16 + 4 stride + 4 bytes each
    assert len(set(calls)) == n_sets    # every set is used (each has its own output buffer)


def test_readout_rotation_explicit_and_large_batches(monkeypatch):
    _fake_cuda(monkeypatch, 126 * 1024 * 1024)
    lib = types.SimpleNamespace(readout_decide=lambda *a: None)
    r = bench.measure_readout(lib, torch, torch.device("cpu"), _Stream(), reps=4, n_sets=3, warmup=1,
                              n_questions=1000, timing_forms=True)
    assert r[4][0] == 3
    # a batch larger than L2 still keeps two sets in turn
    r = bench.measure_readout(lib, torch, torch.device("cpu"), _Stream(), reps=2, warmup=1,
                              n_questions=4_194_304, timing_forms=True)
    assert r[4][0] == 2
