"""The C-ABI library loads and exports every entry point include/*.h declares;
the Python structs match the C layout (CPU only: no compute calls)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import router_softmax_top_gb300 as moe
from router_softmax_top_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 12
    assert declared == set(moe.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == declared


def test_host_only_calls(lib):
    assert moe.moe_expert_bytes(2816, 704) == 3_345_408
    assert moe.moe_expert_bytes(256, 512) == 221_184
    assert moe.moe_expert_bytes(4096, 1536) == 10_616_832
    assert moe.strerror(moe.MOE_OK) == "ok"
    assert "poisoned" in moe.strerror(moe.MOE_ERR_POISONED)
    # null handles are rejected without touching a device
    assert lib.moe_layer_forward(None, 0, None, None, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_cache_sync(None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_cache_launch_count(None) == 0
    n = ctypes.c_uint64(0)
    assert lib.moe_cache_state_size(None, ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_cache_usage(None, None) == moe.MOE_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(64)
    assert lib.moe_cache_save_state(None, buf, 64) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_cache_load_state(None, buf, 64, None) == moe.MOE_ERR_INVALID_ARG
    lib.moe_cache_destroy(None)


def test_init_rejects_bad_config_before_any_cuda_call(lib):
    store = moe.MoeHostStore(None, 0, 0, 0)
    h = ctypes.c_void_p()
    bad = moe.MoeCacheConfig(1, 8, 9, 256, 512, 4, 4, 0, 0, 0, 0, 0, 0, 0, 1000)  # k > E
    assert lib.moe_cache_init(ctypes.byref(bad), ctypes.byref(store), None, ctypes.byref(h)) \
        == moe.MOE_ERR_INVALID_ARG
    bad = moe.MoeCacheConfig(1, 8, 2, 250, 512, 4, 4, 0, 0, 0, 0, 0, 0, 0, 1000)  # H not a multiple of 64
    assert lib.moe_cache_init(ctypes.byref(bad), ctypes.byref(store), None, ctypes.byref(h)) \
        == moe.MOE_ERR_UNSUPPORTED
    for policy, sticky in ((moe.MOE_POLICY_SCORE, 1001), (moe.MOE_POLICY_SCORE, -1),
                           (moe.MOE_POLICY_LRU, 300), (moe.MOE_POLICY_ADOPT, 300), (3, 0)):
        bad = moe.MoeCacheConfig(1, 8, 2, 256, 512, 4, 1, 0, 0, 1, 0, policy, 0, sticky, 1000)
        assert lib.moe_cache_init(ctypes.byref(bad), ctypes.byref(store), None, ctypes.byref(h)) \
            == moe.MOE_ERR_INVALID_ARG, (policy, sticky)
    good = moe.MoeCacheConfig(1, 8, 2, 256, 512, 4, 4, 0, 0, 0, 0, 0, 0, 0, 1000)
    assert lib.moe_cache_init(ctypes.byref(good), ctypes.byref(store), None, ctypes.byref(h)) \
        == moe.MOE_ERR_HOST_STORE   # null store
    assert not h.value


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "moe_cache.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(moe_cache_config), offsetof(moe_cache_config, timeout_us),
         sizeof(moe_host_store), sizeof(moe_cache_stats_t));
  printf("%zu %zu %zu\n", offsetof(moe_cache_stats_t, poisoned), offsetof(moe_cache_stats_t, last_error),
         offsetof(moe_cache_stats_t, cuda_error));
  printf("%zu %zu %zu %u\n", sizeof(moe_cache_state_header), offsetof(moe_cache_state_header, expert_bytes),
         offsetof(moe_cache_state_header, total_bytes), MOE_STATE_MAGIC);
  return 0;
}''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    a, b, c = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines()
    a = [int(v) for v in a.split()]
    b = [int(v) for v in b.split()]
    assert a == [ctypes.sizeof(moe.MoeCacheConfig), moe.MoeCacheConfig.timeout_us.offset,
                 ctypes.sizeof(moe.MoeHostStore), ctypes.sizeof(moe.MoeCacheStats)]
    assert b == [moe.MoeCacheStats.poisoned.offset, moe.MoeCacheStats.last_error.offset,
                 moe.MoeCacheStats.cuda_error.offset]
    assert [int(v) for v in c.split()] == [48, moe.MoeStateHeader.expert_bytes.offset,
                                           moe.MoeStateHeader.total_bytes.offset, moe.MOE_STATE_MAGIC]
    assert ctypes.sizeof(moe.MoeStateHeader) == 48
