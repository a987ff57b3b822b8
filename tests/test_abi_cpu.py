"""The C-ABI library loads, exports every symbol include/gdn.h declares, and
rejects bad arguments on the host before any CUDA call.  No GPU needed: every
call here either is a host-only helper or fails validation."""
import ctypes
import json
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from linear_attention_serving_gdn_gb300 import _build
    _build.build()
    import linear_attention_serving_gdn_gb300 as gdn
    return gdn.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("gdn_prefill_varlen", "gdn_decode_packed", "gdn_mixed_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import linear_attention_serving_gdn_gb300 as gdn
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gdn.h but not exported"
    assert set(declared_functions()) == set(gdn.EXPORTED_SYMBOLS)


def test_prefix_grid_helpers_match_the_page(lib):
    import linear_attention_serving_gdn_gb300 as gdn
    ex = json.load(open(os.path.join(ROOT, "tests", "golden", "prefix_grid.json")))
    assert gdn.gdn_align_block_size(ex["block_size_in"]) == ex["block_size_aligned"]
    assert gdn.gdn_grid_emit_every_chunks(ex["block_size_in"]) == ex["grid"] // ex["chunk"]
    for h in ex["hits"]:
        assert gdn.gdn_floor_prefix_hit(h["hit"], h["prompt"], ex["block_size_in"]) == h["floored"]
    assert gdn.gdn_floor_prefix_hit(2000, 2000, 1056) == 2000
    assert gdn.gdn_align_block_size(0) == -1
    assert gdn.gdn_floor_prefix_hit(5, 4, 1056) == -1


def test_emit_counts_and_offsets(lib):
    import linear_attention_serving_gdn_gb300 as gdn
    cu = [0, 1088, 1088 + 2175, 1088 + 2175 + 32768, 1088 + 2175 + 32768 + 5]
    assert gdn.gdn_prefill_num_emits(cu, 17) == 1 + 1 + 30 + 0
    assert gdn.gdn_prefill_emit_offsets(cu, 17) == [0, 1, 2, 32, 32]
    assert gdn.gdn_prefill_num_emits(cu, 1) == 17 + 33 + 512 + 0
    assert gdn.gdn_prefill_num_emits(cu, 0) == 0
    with pytest.raises(ValueError):
        gdn.gdn_prefill_num_emits([0, 5, 3], 1)


def _Dims(*a):
    from linear_attention_serving_gdn_gb300 import Dims
    return Dims(*a)


FAKE = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: validation fails first


def _decode(lib, dims, rows=4, q=FAKE, src=FAKE, state=FAKE):
    return lib.gdn_decode_packed(ctypes.byref(dims), rows, q, FAKE, FAKE, FAKE, FAKE, state, 8,
                                 src, None, FAKE, None, None)


def test_decode_rejects_bad_arguments_on_the_host(lib):
    ok = _Dims(16, 16, 128, 128, 1.0)
    assert _decode(lib, _Dims(16, 16, 96, 96, 1.0)) == 2          # unsupported head dim
    assert _decode(lib, _Dims(16, 16, 128, 64, 1.0)) == 2         # d_k != d_v
    assert _decode(lib, _Dims(16, 24, 128, 128, 1.0)) == 1        # h_v % h_k != 0
    assert _decode(lib, ok, rows=-1) == 1
    assert _decode(lib, ok, q=None) == 1
    assert _decode(lib, ok, src=None) == 1
    assert _decode(lib, ok, state=ctypes.c_void_p(0x10004)) == 1   # misaligned
    assert lib.gdn_decode_packed(None, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE, None, FAKE,
                                 None, None) == 1
    assert _decode(lib, ok, rows=0) == 0                           # empty: no-op


def _multi(lib, dims, rows=4, T=3, q=FAKE, src=FAKE, state=FAKE):
    return lib.gdn_decode_multi(ctypes.byref(dims), rows, T, q, FAKE, FAKE, FAKE, FAKE, state, 8,
                                src, None, FAKE, None, None)


def test_decode_multi_rejects_bad_arguments_on_the_host(lib):
    ok = _Dims(16, 16, 128, 128, 1.0)
    assert _multi(lib, _Dims(16, 16, 96, 96, 1.0)) == 2
    assert _multi(lib, ok, T=0) == 1                               # at least one token per row
    assert _multi(lib, ok, T=-2) == 1
    assert _multi(lib, ok, rows=-1) == 1
    assert _multi(lib, ok, rows=1 << 20, T=1 << 12) == 2          # rows * T beyond int32
    assert _multi(lib, ok, q=None) == 1
    assert _multi(lib, ok, src=None) == 1
    assert _multi(lib, ok, state=ctypes.c_void_p(0x10008)) == 1   # misaligned
    assert _multi(lib, ok, rows=0) == 0                            # empty: no-op


def test_input_prep_entries_reject_bad_arguments_on_the_host(lib):
    ok = _Dims(16, 16, 128, 128, 1.0)
    prep = lambda T=8, eps=1e-6, q=FAKE, A=FAKE: lib.gdn_prep_inputs(
        ctypes.byref(ok), T, q, FAKE, FAKE, FAKE, A, FAKE, ctypes.c_float(eps), FAKE, FAKE, FAKE, FAKE, None)
    assert prep(T=-1) == 1
    assert prep(eps=-1.0) == 1
    assert prep(q=None) == 1
    assert prep(A=None) == 1
    assert prep(T=0) == 0
    raw = lambda eps=1e-6, a=FAKE: lib.gdn_decode_packed_raw(
        ctypes.byref(ok), 4, FAKE, FAKE, FAKE, a, FAKE, FAKE, FAKE, ctypes.c_float(eps), FAKE, 8, FAKE, None,
        FAKE, None, None)
    assert raw(a=None) == 1
    assert raw(eps=float("nan")) == 1
    assert lib.gdn_decode_packed_raw(ctypes.byref(_Dims(16, 16, 96, 96, 1.0)), 4, FAKE, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, FAKE, ctypes.c_float(1e-6), FAKE, 8, FAKE, None, FAKE, None,
                                     None) == 2


def _prefill(lib, cu_host, n, E=0, cap=0, cs=None, dims=None, ws=None, ws_bytes=0):
    dims = dims or _Dims(16, 32, 128, 128, 1.0)
    arr = (ctypes.c_int32 * len(cu_host))(*cu_host)
    return lib.gdn_prefill_varlen(ctypes.byref(dims), n, FAKE, arr, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, 8, None, None, FAKE, cs, E, cap, ws, ws_bytes, None, None)


def test_prefill_rejects_bad_arguments_on_the_host(lib):
    assert _prefill(lib, [0, 10, 5], 2) == 1                       # non-monotone
    assert _prefill(lib, [3, 10], 1) == 1                          # does not start at 0
    assert _prefill(lib, [0, 2000], 1, E=1, cap=30, cs=FAKE) == 1  # 31 emits needed
    assert _prefill(lib, [0, 2000], 1, E=1, cap=31, cs=None) == 1  # stream missing
    assert _prefill(lib, [0, 2000], 1, E=-1) == 1
    assert _prefill(lib, [0, 10], 1, dims=_Dims(16, 32, 256, 256, 1.0)) == 2
    assert _prefill(lib, [0, 2000], 1, E=(1 << 24) + 1, cap=1, cs=FAKE) == 1  # 64 E beyond int32 range
    assert _prefill(lib, [0], 0) == 0                              # no sequences: no-op


def test_prefill_workspace_contract(lib):
    import linear_attention_serving_gdn_gb300 as gdn
    dims = _Dims(16, 32, 128, 128, 1.0)
    need = lib.gdn_prefill_workspace_bytes(ctypes.byref(dims), 8, 4901)
    assert need == gdn.gdn_prefill_workspace_bytes(16, 32, 128, 8, 4901)
    assert lib.gdn_prefill_workspace_bytes(ctypes.byref(_Dims(16, 32, 96, 96, 1.0)), 8, 10) == ctypes.c_size_t(-1).value
    assert lib.gdn_prefill_workspace_bytes(ctypes.byref(dims), -1, 10) == ctypes.c_size_t(-1).value
    # A workspace must be 256-byte aligned and at least `need` bytes; both are
    # checked on the host before anything is launched (GDN_ERR_WORKSPACE).
    assert _prefill(lib, [0, 10], 1, ws=ctypes.c_void_p(0x10010), ws_bytes=1 << 20) == 4
    if need > 0:
        assert _prefill(lib, [0, 10], 1, ws=ctypes.c_void_p(0x10000), ws_bytes=need - 1) == 4
        assert _prefill(lib, [0, 10], 1) == 4
    for bad_dims in (_Dims(16, 32, 64, 128, 1.0), _Dims(16, 24, 128, 128, 1.0)):
        assert _prefill(lib, [0, 10], 1, dims=bad_dims, ws=ctypes.c_void_p(0x10010)) in (1, 2)


def _apc(lib, cu_host, n, E=17, table=FAKE, stride=4, first=FAKE, state=FAKE):
    dims = _Dims(16, 32, 128, 128, 1.0)
    arr = (ctypes.c_int32 * len(cu_host))(*cu_host)
    return lib.gdn_prefill_varlen_apc(ctypes.byref(dims), n, FAKE, arr, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      state, 8, None, None, FAKE, E, table, stride, first, None, 0, None,
                                      None)


def test_prefill_apc_rejects_bad_arguments_on_the_host(lib):
    assert _apc(lib, [0, 2000], 1, E=0) == 1                       # a block size is required
    assert _apc(lib, [0, 2000], 1, table=None) == 1
    assert _apc(lib, [0, 2000], 1, first=None) == 1
    assert _apc(lib, [0, 2000], 1, stride=0) == 1
    assert _apc(lib, [0, 2000], 1, state=None) == 1
    assert _apc(lib, [0, 10, 5], 2) == 1                           # non-monotone
    assert _apc(lib, [0], 0) == 0                                  # no sequences: no-op


def _mixed(lib, dims, nd, n_p, cu, dec_src=FAKE, cs=None, E=0, cap=0, ws=None):
    return lib.gdn_mixed_step(ctypes.byref(dims), nd, n_p, FAKE, cu, FAKE, FAKE, FAKE, FAKE, FAKE,
                              FAKE, 8, dec_src, None, None, None, FAKE, cs, E, cap, ws, 0, None, None)


def test_mixed_step_rejects_bad_arguments_on_the_host(lib):
    dims = _Dims(16, 16, 128, 128, 1.0)
    bad = (ctypes.c_int32 * 3)(0, 7, 2)
    assert _mixed(lib, dims, 4, 2, bad) == 1
    good = (ctypes.c_int32 * 2)(0, 7)
    assert _mixed(lib, dims, -1, 1, good) == 1
    assert _mixed(lib, dims, 4, 1, good, dec_src=None) == 1


def test_mixed_step_validates_the_prefill_half_before_launching_decode(lib):
    # Valid decode rows but a bad prefill half: the call must fail validation
    # (1 or 4) before the decode kernel is launched.  Without a GPU a launch
    # would have returned GDN_ERR_CUDA (3) instead.
    dims = _Dims(16, 16, 128, 128, 1.0)
    cu = (ctypes.c_int32 * 2)(0, 2000)
    assert _mixed(lib, dims, 4, 1, cu, cs=ctypes.c_void_p(0x10008), E=1, cap=31) == 1  # misaligned stream
    assert _mixed(lib, dims, 4, 1, cu, cs=FAKE, E=1, cap=30) == 1                       # 31 emits needed
    assert _mixed(lib, dims, 4, 1, cu, E=(1 << 24) + 1) == 1                            # emission stride
    assert _mixed(lib, dims, 4, 1, cu, ws=ctypes.c_void_p(0x10010)) == 4               # workspace alignment


def _colaunch(lib, dims, nd, n_p, cu, aux=FAKE, fork=FAKE, join=FAKE, cs=None, E=0, cap=0):
    return lib.gdn_mixed_step_colaunch(ctypes.byref(dims), nd, n_p, FAKE, cu, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       FAKE, 8, FAKE, None, None, None, FAKE, cs, E, cap, None, 0, None,
                                       None, aux, fork, join)


def test_mixed_step_colaunch_validates_before_forking(lib):
    # A separate decode stream needs both events; a bad half of the step is
    # rejected before any event is recorded or kernel launched (either would
    # have returned GDN_ERR_CUDA without a GPU).
    dims = _Dims(16, 16, 128, 128, 1.0)
    cu = (ctypes.c_int32 * 2)(0, 2000)
    assert _colaunch(lib, dims, 4, 1, cu, fork=None) == 1
    assert _colaunch(lib, dims, 4, 1, cu, join=None) == 1
    assert _colaunch(lib, dims, 4, 1, cu, cs=FAKE, E=1, cap=30) == 1      # 31 emits needed
    assert _colaunch(lib, dims, -1, 1, cu) == 1
    bad = (ctypes.c_int32 * 3)(0, 7, 2)
    assert _colaunch(lib, dims, 4, 2, bad) == 1


def test_status_from_device_word(lib):
    import linear_attention_serving_gdn_gb300 as gdn
    assert gdn.gdn_status_from_device(0) == 0
    assert gdn.gdn_status_from_device(gdn.GDN_DEV_TIMEOUT) == 5
    assert gdn.gdn_status_from_device(gdn.GDN_DEV_TIMEOUT | gdn.GDN_DEV_BAD_SLOT) == 5
    assert gdn.gdn_status_from_device(gdn.GDN_DEV_BAD_SLOT) == 1
    assert "workspace" in gdn.gdn_status_string(4)
    assert "wait" in gdn.gdn_status_string(5)


def test_status_strings(lib):
    import linear_attention_serving_gdn_gb300 as gdn
    assert gdn.gdn_status_string(0) == "GDN_OK"
    assert "invalid" in gdn.gdn_status_string(1)
