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
    assert a.preload_profile == 0 and a.preload_from_session == 0   # cold start unless asked
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


def test_profiled_figures_follow_the_kernel_source(tmp_path, monkeypatch):
    # ncu figures (traffic ratio, instructions per weight) are used while the
    # kernel's source text is the one captured, and dropped once it changes
    import hashlib
    import json
    csrc = tmp_path / "router_softmax_top_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = "head\n<<kernel body>>\ntail\n"
    (csrc / "k.cu").write_text(src)
    body = src[src.find("<<"):src.find(">>")]
    entry = {"file": "k.cu", "begin": "<<", "end": ">>",
             "source_sha256": hashlib.sha256(body.encode()).hexdigest(),
             "dram_bytes_per_algorithmic_byte": 1.01, "warp_inst_per_weight": 0.2}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_entry("k")["warp_inst_per_weight"] == 0.2
    assert bench.profiled_traffic_ratio("k") == 1.01
    assert bench.profiled_entry("absent") is None
    (csrc / "k.cu").write_text(src.replace("body", "b0dy"))
    assert bench.profiled_entry("k") is None and bench.profiled_traffic_ratio("k") is None


def test_committed_decode_figures_match_the_kernel():
    # the committed capture is of the decode layer kernel as it stands
    e = bench.profiled_entry("decode_layer")
    assert e is not None, "decode_layer_kernel changed since profiles/traffic.json was captured"
    assert 1.0 <= e["dram_bytes_per_algorithmic_byte"] < 1.05 and 0 < e["warp_inst_per_weight"] < 1
