"""The C ABI on a machine without a GPU: the library loads, exports every
entry point that include/moe.h declares, and rejects bad arguments before any
CUDA work."""

import ctypes as C
import os
import re
import subprocess

import pytest

import bit_routed_expert_router_gb300 as moe
from bit_routed_expert_router_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def declared_functions():
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("moe_create", "moe_init_layer", "moe_set_slots", "moe_decode_step", "moe_prefill", "moe_destroy",
              "moe_route_noalloc"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", moe_build.SO], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        getattr(lib, n)


def test_binding_wraps_every_declared_function(lib):
    for n in declared_functions():
        assert hasattr(moe, n), f"binding lacks {n}"


def test_expert_sizes(lib):
    cfg = moe.make_config(2816, 704, 2816, 128, 8)
    assert moe.moe_expert_bytes(cfg) == 3_345_408
    assert moe.moe_shared_bytes(cfg) == 13_381_632
    tiny = moe.make_config(256, 128, 128, 8, 2)
    assert moe.moe_expert_bytes(tiny) == 55_296


@pytest.mark.parametrize("kw", [dict(d=250), dict(f=100), dict(f_shared=0), dict(n_experts=0), dict(n_experts=300),
                                dict(top_k=0), dict(top_k=9), dict(d=4096), dict(max_tokens=0)])
def test_bad_configs_are_rejected_before_cuda(lib, kw):
    base = dict(d=256, f=128, f_shared=128, n_experts=8, top_k=2)
    base.update(kw)
    cfg = moe.make_config(base["d"], base["f"], base["f_shared"], base["n_experts"], base["top_k"],
                          max_tokens=kw.get("max_tokens", 32))
    st, h = moe.moe_create(cfg, 0)
    assert st == moe.MOE_EINVAL and h is None
    assert moe.moe_last_error(None)
    assert moe.moe_expert_bytes(cfg) == 0


def test_null_context_is_rejected(lib):
    assert lib.moe_set_slots(None, 4) == moe.MOE_EINVAL
    assert lib.moe_reset_cache(None) == moe.MOE_EINVAL
    assert lib.moe_set_cache_policy(None, 1) == moe.MOE_EINVAL
    assert lib.moe_sync(None, None) == moe.MOE_EINVAL
    assert lib.moe_profile(None, 1) == moe.MOE_EINVAL
    assert lib.moe_test_hook(None, 1, 0) == moe.MOE_EINVAL
    assert lib.moe_set_debug(None, None, None, None, None, 0) == moe.MOE_EINVAL
    assert lib.moe_set_expert_file(None, b"/nonexistent/e.bin", 4, 0, 0) == moe.MOE_EINVAL
    assert lib.moe_set_file_cache(None, 8) == moe.MOE_EINVAL
    assert lib.moe_set_staging(None, moe.MOE_STAGING_DEVICE) == moe.MOE_EINVAL
    assert lib.moe_decode_step(None, None, 1, 0, 1, None, None, None, None, 0, None, None) == moe.MOE_EINVAL
    assert lib.moe_prefill(None, None, 1, 0, 1, None, None, None, None) == moe.MOE_EINVAL
    st = moe.MoeStats()
    assert lib.moe_get_stats(None, C.byref(st)) == moe.MOE_EINVAL
    lib.moe_destroy(None)


def test_noalloc_routing_rejects_bad_sizes_without_cuda(lib):
    cfg = moe.make_config(256, 128, 128, 8, 2)
    assert moe.moe_route_noalloc(cfg, 16, 16, 0, None, 16, 16, 0) == moe.MOE_EINVAL
    assert moe.moe_route_noalloc(cfg, 16, 16, moe.ROUTE_NOALLOC_MAX_B + 1, None, 16, 16, 0) == moe.MOE_EINVAL
    assert moe.moe_route_noalloc(cfg, None, 16, 1, None, 16, 16, 0) == moe.MOE_EINVAL


def test_host_read_rate_rejects_bad_arguments_without_cuda(lib):
    out = C.c_double(1.0)
    assert lib.moe_host_read_rate(None, 1024, 1, None, C.byref(out)) == moe.MOE_EINVAL
    buf = (C.c_uint8 * 1024)()
    assert lib.moe_host_read_rate(buf, 1000, 1, None, C.byref(out)) == moe.MOE_EINVAL     # not a multiple of 16
    assert lib.moe_host_read_rate(buf, 1024, 0, None, C.byref(out)) == moe.MOE_EINVAL     # no repetition
    assert lib.moe_host_read_rate(buf, 1024, 1, None, None) == moe.MOE_EINVAL


def test_status_strings(lib):
    for i, name in enumerate(["MOE_OK", "MOE_EINVAL", "MOE_ENOMEM", "MOE_ECUDA", "MOE_ESTATE", "MOE_ETIMEOUT",
                              "MOE_EDOMAIN"]):
        assert moe.status_name(i) == name
