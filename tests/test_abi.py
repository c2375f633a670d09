"""The C-ABI library builds, loads without a GPU, and exports every entry
point include/moe.h declares; host-side argument checks (no device work)."""
import ctypes
import os
import re

import pytest

from routed_mixture_experts_router_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared():
    src = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def test_header_lists_entry_points():
    names = declared()
    assert sorted(names) == sorted(binding.ENTRY_POINTS)


def test_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert "sm_103a" in binding.version()


def _layer(E=128, k=8, d=2048, f=768, ptr=0x10000):
    q = binding.Q8Mat(ptr, ptr)
    return binding.LayerW(E, k, d, f, q, q, q, ptr, 0)


def test_workspace_size(lib):
    w = _layer()
    T = 1024
    n = lib.moe_workspace_size(T, ctypes.byref(w), 0, 0)
    P = T * 8
    # routing (idx, wts), offsets, three pair arrays, h fp32 [P][d_ff]
    assert n >= P * 4 * 5 + 129 * 4 + P * 768 * 4
    assert n % 256 == 0
    n_det = lib.moe_workspace_size(T, ctypes.byref(w), 0, binding.MOE_FLAG_DETERMINISTIC)
    assert n_det >= n + P * 2048 * 4
    assert lib.moe_workspace_size(T, ctypes.byref(_layer(k=0)), 0, 0) == 0
    assert lib.moe_workspace_size(T, ctypes.byref(_layer(E=300)), 0, 0) == 0
    assert lib.moe_workspace_size(T, ctypes.byref(_layer(d=2050)), 0, 0) == 0
    assert lib.moe_workspace_size(-1, ctypes.byref(w), 0, 0) == 0


@pytest.mark.parametrize("bad", [dict(k=9, E=8), dict(k=33, E=64), dict(d=100), dict(f=0), dict(E=0)])
def test_invalid_geometry_rejected_on_host(lib, bad):
    w = _layer(**bad)
    P = ctypes.c_void_p(0x10000)
    assert lib.moe_route(P, 4, ctypes.byref(w), P, P, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(P, 4, ctypes.byref(w), 0, 0, 0, ctypes.c_void_p(0x20000), None, None, None, P,
                                 1 << 30, None, None) == binding.MOE_ERR_INVALID_ARG


def test_invalid_pointers_rejected_on_host(lib):
    w = _layer()
    good = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10004)
    assert lib.moe_route(mis, 4, ctypes.byref(w), good, good, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, 4, ctypes.byref(w), good, good, None) == binding.MOE_ERR_INVALID_ARG
    # out aliasing x
    assert lib.moe_layer_forward(good, 4, ctypes.byref(w), 0, 0, 0, good, None, None, None, good, 1 << 30, None,
                                 None) == binding.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned
    assert lib.moe_layer_forward(good, 4, ctypes.byref(w), 0, 0, 0, ctypes.c_void_p(0x20000), None, None, None,
                                 good, 16, None, None) == binding.MOE_ERR_WORKSPACE
    assert lib.moe_layer_forward(good, 4, ctypes.byref(w), 0, 0, 0, ctypes.c_void_p(0x20000), None, None, None,
                                 ctypes.c_void_p(0x10010), 1 << 30, None, None) == binding.MOE_ERR_WORKSPACE
    assert lib.moe_pack_q8(good, 4, 33, good, good, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_bucket(good, 4, 9, 8, good, good, good, good, None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(good, good, good, 4, 2, 100, None, good, None) == binding.MOE_ERR_INVALID_ARG


def test_empty_batch_is_ok_without_device_work(lib):
    w = _layer()
    assert lib.moe_route(None, 0, ctypes.byref(w), None, None, None) == binding.MOE_OK
    assert lib.moe_layer_forward(None, 0, ctypes.byref(w), 0, 0, 0, None, None, None, None, None, 0, None,
                                 None) == binding.MOE_OK


def test_binding_fails_loudly_without_library(tmp_path):
    saved = binding._lib
    try:
        binding._lib = None
        with pytest.raises(RuntimeError):
            binding.load(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved


def test_arena_sizes(lib):
    """Blob bytes: a 4 KiB header page + the expert's payload, page-rounded
    (the pages' 5,017,600 B per Q8_0 expert of the qwen3_moe geometry)."""
    w = _layer()
    assert lib.moe_arena_blob_bytes(ctypes.byref(w)) == 5_017_600
    w.wfmt = binding.MOE_WFMT_Q4_0
    assert lib.moe_arena_blob_bytes(ctypes.byref(w)) == 4096 + 2_654_208     # 648 whole pages
    w.wfmt = 2
    assert lib.moe_arena_blob_bytes(ctypes.byref(w)) == 0
    n = lib.moe_arena_state_bytes(48, 128, 1536)
    assert n >= 64 + 48 * 128 * 4 + 2 * 1536 * 4 + 2 * 128 * 4 and n % 256 == 0
    assert lib.moe_arena_state_bytes(0, 128, 1536) == 0
    assert lib.moe_arena_state_bytes(48, 300, 1536) == 0
    assert lib.moe_arena_state_bytes(48, 128, 70000) == 0


def test_arena_argument_checks(lib):
    """Refused on the host before any device work."""
    P = ctypes.c_void_p
    fake = P(0x10000)
    assert lib.moe_arena_init(None, 48, 128, 1536, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_arena_init(P(0x10010), 48, 128, 1536, None) == binding.MOE_ERR_INVALID_ARG  # not 256-aligned
    w = _layer()
    w.n_slots = 1536
    assert lib.moe_arena_admit(None, 0, fake, 8, fake, ctypes.byref(w), fake, None, None) == \
        binding.MOE_ERR_INVALID_ARG
    assert lib.moe_arena_admit(fake, 0, fake, 8, P(0x10008), ctypes.byref(w), fake, None, None) == \
        binding.MOE_ERR_INVALID_ARG                                                            # blobs misaligned
    w.n_slots = 0
    assert lib.moe_arena_admit(fake, 0, fake, 8, fake, ctypes.byref(w), fake, None, None) == \
        binding.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_arena(fake, 1, ctypes.byref(w), 0, 0, 0, P(0x20000), fake, 0, fake, fake,
                                       1 << 20, None, None) == binding.MOE_ERR_INVALID_ARG
    w.expert_slot = 0x30000                     # a slot map needs 1..65536 slots
    assert lib.moe_workspace_size(4, ctypes.byref(w), 0, 0) > 0
    assert lib.moe_layer_forward(fake, 4, ctypes.byref(w), 0, 0, 0, P(0x20000), None, None, None, fake, 1 << 30,
                                 None, None) == binding.MOE_ERR_INVALID_ARG


def test_q4_geometry_refused(lib):
    """Q4_0 needs d_model % 512 == 0 (its kernels' K split): d_model 256 is
    refused as unsupported before any device work."""
    w = _layer(E=16, k=2, d=256, f=128)
    w.wfmt = binding.MOE_WFMT_Q4_0
    P = ctypes.c_void_p
    assert lib.moe_layer_forward(P(0x10000), 4, ctypes.byref(w), 0, 0, 0, P(0x20000), None, None, None,
                                 P(0x40000), 1 << 30, None, None) == binding.MOE_ERR_UNSUPPORTED


def test_arena_blob_matches_printed_cache_sizes(lib):
    """The library's blob for a Q8_0 expert of the qwen3_moe geometry
    reproduces the pages' printed raw-cache sizes for every slot count and
    their bytes per miss (tests/golden/expert_cache_sizes.txt)."""
    blob = lib.moe_arena_blob_bytes(ctypes.byref(_layer()))
    rows = [ln.split() for ln in open(os.path.join(ROOT, "tests", "golden", "expert_cache_sizes.txt"))
            if ln.strip() and not ln.startswith("#")]
    checked = 0
    for kind, *vals in rows:
        if kind == "raw_cache_gib":
            assert round(int(vals[0]) * blob / 2 ** 30, 2) == float(vals[1]), vals
            checked += 1
        elif kind == "miss_bytes":
            per_miss = float(vals[1]) * 1e9 / int(vals[0])
            assert abs(per_miss - blob) / blob < 3e-3, vals
            checked += 1
    assert checked == 6
