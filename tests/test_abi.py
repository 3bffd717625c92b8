"""The C ABI of libsanta.so, checked without a GPU: the library loads, exports every
symbol include/santa.h declares, sizes workspaces, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

from stochastic_sparse_kv_gb300 import santa, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return santa.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "santa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(santa_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(santa.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert santa.status_string(0) == "ok"
    for rc in (-1, -2, -3, -4, -5, -6):
        assert santa.status_string(rc) not in ("ok", "unknown status")
    assert lib.santa_version() >= 10000


def test_workspace_size_matches_layout(lib):
    sh = santa.make_shape(16, 32, 8, 128, 32768)
    n = santa.workspace_size(sh, 256, "systematic")
    # w fp32 per (b, h_q, key) dominates: 16*32*32768*4 = 67 MB
    assert 16 * 32 * 32768 * 4 < n < 16 * 32 * 32768 * 4 * 1.2
    nd = santa.workspace_size(sh, 1, "dense")
    # dense: one partial (o, m, l) per query head and 512-key unit
    assert nd >= 16 * 32 * (32768 // 512) * (128 + 2) * 4
    assert n % 256 == 0 and nd % 256 == 0


@pytest.mark.parametrize("shape,S,mode,rc", [
    ((16, 32, 8, 128, 32768), 256, 2, 0),
    ((0, 32, 8, 128, 32768), 256, 2, -1),       # B < 1
    ((1, 30, 8, 128, 1024), 256, 2, -1),        # H_q % H_kv != 0
    ((1, 48, 3, 128, 1024), 256, 2, -4),        # G = 16 unsupported
    ((1, 32, 8, 96, 1024), 256, 2, -4),         # d = 96 unsupported
    ((1, 32, 8, 128, 1024), 0, 2, -1),          # S = 0
    ((1, 32, 8, 128, 1024), 4097, 1, -1),       # S too large
    ((1, 32, 8, 128, 1024), 0, 0, 0),           # dense ignores S
    ((1, 32, 8, 128, 1024), 16, 7, -1),         # bad mode
    ((1, 32, 8, 128, 1024), 16, 0x102, 0),      # SANTA_GROUP_DEDUP is a valid flag
    ((1, 32, 8, 128, 1024), 16, 0x202, 0),      # SANTA_OUT_BF16 is a valid flag
    ((1, 32, 8, 128, 1024), 16, 0x302, 0),      # both flags
    ((1, 32, 8, 128, 1024), 16, 0x402, 0),      # SANTA_BERNOULLI_QK is a valid flag
    ((1, 32, 8, 128, 1024), 16, 0x400, 0),      # ... also with the dense mode
    ((1, 32, 8, 128, 1024), 16, 0x802, 0),      # SANTA_TWO_PASS is a valid flag
    ((1, 32, 8, 128, 1024), 16, 0x1002, -1),    # unknown flag bits
    ((1025, 32, 8, 128, 1024), 16, 2, -4),      # B > 1024
    ((1, 32, 8, 128, 524289), 16, 2, -4),       # n_max too large
    ((1024, 8, 8, 64, 262144), 16, 2, -4),      # B*H_kv*n_max = 2^31 cache rows: past 32-bit copy coordinates
    ((1024, 8, 8, 64, 262143), 16, 0, 0),       # one row short of it (dense)
])
def test_workspace_size_validation(lib, shape, S, mode, rc):
    sh = santa.make_shape(*shape)
    n = ctypes.c_size_t(0)
    assert lib.santa_workspace_size(ctypes.byref(sh), S, mode, ctypes.byref(n)) == rc


def test_decode_rejects_bad_arguments_on_the_host(lib):
    sh = santa.make_shape(1, 4, 1, 64, 256)
    good = 4096  # a fake, 256-aligned address: never dereferenced, validation comes first
    ws_n = santa.workspace_size(sh, 16, 2)
    args = dict(q=good, k=good, v=good, sl=good, S=16, mode=2, out=good, idx=good, ws=good, wsn=ws_n)

    def call(**kw):
        a = {**args, **kw}
        return lib.santa_decode(ctypes.byref(sh), ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]),
                                ctypes.c_void_p(a["v"]), ctypes.c_void_p(a["sl"]), a["S"], a["mode"],
                                ctypes.c_uint64(0), ctypes.c_void_p(a["out"]), ctypes.c_void_p(a["idx"]),
                                ctypes.c_void_p(a["ws"]), a["wsn"], None)

    assert call(q=0) == -1
    assert call(sl=0) == -1
    assert call(out=0) == -1
    assert call(ws=0) == -3
    assert call(wsn=ws_n - 1) == -3
    assert call(q=good + 8) == -2
    assert call(ws=good + 16) == -2
    assert call(S=0) == -1
    assert call(mode=9) == -1
    bad = santa.make_shape(1, 4, 3, 64, 256)
    assert lib.santa_decode(ctypes.byref(bad), None, None, None, None, 16, 2, ctypes.c_uint64(0),
                            None, None, None, 0, None) == -1
    assert lib.santa_sample_points(0, 1, 1, 2, ctypes.c_uint64(0), ctypes.c_void_p(good), None) == -1
    assert lib.santa_sample_points(1, 1, 1, 0, ctypes.c_uint64(0), ctypes.c_void_p(good), None) == -1
    assert lib.santa_ternary_query(0, 1, 128, ctypes.c_void_p(good), ctypes.c_uint64(0), ctypes.c_void_p(good),
                                   None) == -1
    n = ctypes.c_int32(0)
    assert lib.santa_call_info(ctypes.byref(bad), 16, 2, ctypes.byref(n)) == -1
    assert lib.santa_call_info(ctypes.byref(sh), 0, 2, ctypes.byref(n)) == -1
    assert lib.santa_call_info(ctypes.byref(sh), 16, 2, None) == -1
    assert lib.santa_call_info(ctypes.byref(sh), 16, 0x1002, ctypes.byref(n)) == -1
    assert lib.santa_ternary_query(1, 1, 96, ctypes.c_void_p(good), ctypes.c_uint64(0), ctypes.c_void_p(good),
                                   None) == -4
    assert lib.santa_ternary_query(1, 1, 128, ctypes.c_void_p(good + 2), ctypes.c_uint64(0),
                                   ctypes.c_void_p(good), None) == -2


def test_binding_refuses_to_run_without_the_library(tmp_path):
    import importlib
    mod = importlib.reload(santa)
    try:
        with pytest.raises(RuntimeError):
            mod._lib = None
            mod.load(str(tmp_path / "missing.so"))
    finally:
        importlib.reload(santa)


def test_wait_limit_setter_is_host_only(lib):
    # a process-wide setting read by later calls; no device work
    assert lib.santa_set_wait_limit(ctypes.c_uint64(1000)) == 0
    assert lib.santa_set_wait_limit(ctypes.c_uint64(0)) == 0


def test_binding_checks_tensors_before_calling_the_library():
    import torch
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16)
    sl = torch.tensor([256], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        santa.decode(q, k, k, sl, 16, "systematic")          # host tensors
    with pytest.raises(ValueError, match="CUDA"):
        santa.DecodePlan(q, k, k, sl, 16, "dense")
    with pytest.raises(ValueError):
        santa.decode(q.float(), k, k, sl, 16, "systematic")  # wrong dtype


def test_static_entry_point_checks_arguments_before_touching_the_device(lib):
    """santa_decode_static returns argument errors before it enqueues anything: with no GPU
    here, any device call would fail with SANTA_ERR_CUDA instead.  The stream is a bogus
    handle that must never be used."""
    lib = santa.load()  # (an earlier test reloads the binding module)
    sh = santa.make_shape(1, 4, 1, 64, 256)
    good = 4096
    bogus_stream = ctypes.c_void_p(0xDEAD0)

    def call(q=good, out=good, idx=good, S=16, mode=2):
        return lib.santa_decode_static(ctypes.byref(sh), ctypes.c_void_p(q), ctypes.c_void_p(good),
                                       ctypes.c_void_p(good), ctypes.c_void_p(good), S, mode, ctypes.c_uint64(0),
                                       ctypes.c_void_p(out), ctypes.c_void_p(idx), bogus_stream)

    assert call(q=0) == -1
    assert call(out=0) == -1
    assert call(out=good + 4) == -2
    assert call(idx=good + 2) == -2
    assert call(S=0) == -1
    assert call(mode=9) == -1
