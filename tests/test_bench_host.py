"""Host-side logic of bench.py (CPU only): the host store's NUMA binding and the
option defaults the timed runs rely on."""
import ctypes
import mmap
import sys

import pytest

import bench


def test_store_bound_to_node_0_lands_there():
    t = bench.host_store(64 << 20, node=0, strict=True)
    t.numpy()[:] = 1                       # first touch after the binding
    pages = bench.host_store_numa(t)
    if pages is None:
        pytest.skip("no /proc/self/numa_maps")
    assert set(pages) == {"N0"} and pages["N0"] > 0


def test_binding_to_an_absent_node_is_refused():
    mm = mmap.mmap(-1, 1 << 21, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    base = ctypes.addressof(ctypes.c_char.from_buffer(mm))
    assert not bench.bind_to_node(base, 1 << 21, 1000)
    assert not bench.bind_to_node(base, 1 << 21, -1)
    with pytest.raises(SystemExit):
        bench.host_store(1 << 21, node=1000, strict=True)
    bench.host_store(1 << 21, node=1000, strict=False)   # auto mode: first touch instead


def test_defaults(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.resolve_defaults(bench.parse())
    assert (a.gpus, a.impl, a.workload, a.fill, a.policy) == (1, "ours", "decode", "pull", "lru")
    assert a.warmup == bench.DECODE_WARMUP >= bench.COLD_STEPS >= 3 and a.steps >= 1
    for extra in (["--workload", "prefill"], ["--impl", "reference"]):
        monkeypatch.setattr(sys, "argv", ["bench.py"] + extra)
        assert bench.resolve_defaults(bench.parse()).warmup == 64
    monkeypatch.setattr(sys, "argv", ["bench.py", "--warmup", "5"])
    assert bench.resolve_defaults(bench.parse()).warmup == 5
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.store_node == "auto" and a.gemm_min_tokens == 16 and a.tokens == 512
    assert a.preload_profile == 0 and a.decode_after == 0
    monkeypatch.setattr(sys, "argv", ["bench.py", "--store-node", "none"])
    assert bench.store_node(bench.parse()) == -1
    monkeypatch.setattr(sys, "argv", ["bench.py", "--store-node", "3"])
    assert bench.store_node(bench.parse()) == 3


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    # under torchrun only rank 0 times the oracle and prints; rank 1 returns at once
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    assert bench.run_reference(bench.resolve_defaults(bench.parse())) is None
    assert capsys.readouterr().out == ""


def test_cpu_model_names_the_host():
    m = bench.host_cpu_model()
    assert m.endswith(f"{__import__('os').cpu_count()} logical CPUs") and not m.startswith("unknown,")
