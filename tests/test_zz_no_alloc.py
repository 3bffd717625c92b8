"""santa_decode_static: the decode entry point for callers that cannot allocate device
memory (the library supplies the scratch from a fixed device array of
SANTA_STATIC_SCRATCH_BYTES).  Checked through the C ABI against santa_decode with a
caller-owned workspace: bit-identical results on two calls in a row in every mode, calls
of other shapes and modes in between, the device error word, and no device allocation.

The file name makes pytest collect it last, so that a run stopping at the first failure
has already run every other test.  It also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from stochastic_sparse_kv_gb300 import santa, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _call_static(lib, shape, q, k, v, sl, S, mode, seed, out, idx, stream):
    return lib.santa_decode_static(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(sl), S, mode,
                                   ctypes.c_uint64(seed), _ptr(out), _ptr(idx), ctypes.c_void_p(stream))


def _call_workspace(lib, shape, q, k, v, sl, S, mode, seed, out, idx, ws, stream):
    return lib.santa_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(sl), S, mode,
                            ctypes.c_uint64(seed), _ptr(out), _ptr(idx), _ptr(ws), ws.numel(),
                            ctypes.c_void_p(stream))


def _inputs(seq, H_q, H_kv, n_max, S, seed):
    _, q, k, v, sl = workloads.small("static", len(seq), H_q, H_kv, 128, n_max, S, seq_lens=seq, seed=seed)
    return q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)


def _compare(lib, inp, H_kv, n_max, S, mode, seeds):
    """Both entry points on the same inputs: outputs and indices must be identical (same
    kernels, same inputs, deterministic arithmetic)."""
    qd, kd, vd, sld = inp
    B, H_q, d = qd.shape
    shape = santa.make_shape(B, H_q, H_kv, d, n_max)
    stream = torch.cuda.current_stream().cuda_stream
    ws = santa.new_workspace(santa.workspace_size(shape, S, mode), DEV)
    sampled = (mode & 0xff) != santa.DENSE
    for seed in seeds:
        out_a = torch.full((B, H_q, d), float("nan"), device=DEV)
        out_b = torch.full((B, H_q, d), float("nan"), device=DEV)
        idx_a = torch.full((B, H_q, S), -7, dtype=torch.int32, device=DEV) if sampled else None
        idx_b = torch.full((B, H_q, S), -7, dtype=torch.int32, device=DEV) if sampled else None
        assert _call_static(lib, shape, qd, kd, vd, sld, S, mode, seed, out_a, idx_a, stream) == 0
        assert _call_workspace(lib, shape, qd, kd, vd, sld, S, mode, seed, out_b, idx_b, ws, stream) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out_a).all()
        assert torch.equal(out_a, out_b)
        if sampled:
            assert torch.equal(idx_a, idx_b)


@pytest.mark.parametrize("mode", [santa.SYSTEMATIC, santa.STRATIFIED, santa.IID, santa.DENSE,
                                  santa.SYSTEMATIC | santa.GROUP_DEDUP])
def test_static_scratch_matches_workspace_entry_point(mode):
    lib = santa.load()
    inp = _inputs([3000, 777, 0, 2049], 16, 4, 3000, 96, 21)
    _compare(lib, inp, 4, 3000, 96, mode, seeds=(5, 6))  # two calls in a row


def test_static_scratch_after_other_shapes_and_modes():
    """The shared buffer keeps whatever the last call left in it: a large sampled call, a
    dense call and a sampled call of another shape in turn must each still match the
    workspace entry point."""
    lib = santa.load()
    big = _inputs([20000, 12000], 32, 8, 20000, 512, 3)
    _compare(lib, big, 8, 20000, 512, santa.STRATIFIED, seeds=(1,))
    small = _inputs([1500, 999, 1], 8, 2, 1500, 64, 4)
    _compare(lib, small, 2, 1500, 64, santa.DENSE, seeds=(0,))
    _compare(lib, small, 2, 1500, 64, santa.SYSTEMATIC, seeds=(2,))
    _compare(lib, big, 8, 20000, 128, santa.IID, seeds=(3,))


def test_static_scratch_allocates_nothing():
    """After a first call (which looks up the scratch's device address), further calls
    leave the device's free memory exactly unchanged."""
    lib = santa.load()
    qd, kd, vd, sld = _inputs([4096, 2000], 32, 8, 4096, 256, 8)
    shape = santa.make_shape(2, 32, 8, 128, 4096)
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.empty(2, 32, 128, device=DEV)
    idx = torch.empty(2, 32, 256, dtype=torch.int32, device=DEV)
    assert _call_static(lib, shape, qd, kd, vd, sld, 256, santa.SYSTEMATIC, 0, out, idx, stream) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for seed in range(1, 6):
        for mode in (santa.SYSTEMATIC, santa.DENSE):
            assert _call_static(lib, shape, qd, kd, vd, sld, 256, mode, seed, out, idx, stream) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_static_scratch_reports_device_errors():
    """An out-of-range seq_lens on the static path sets the scratch's own error word, which
    santa_device_status(NULL, ...) reads and clears; the next call does not hide it."""
    lib = santa.load()
    _, q, k, v, _ = workloads.small("bad", 2, 8, 2, 128, 512, 16, seq_lens=[512, 300], seed=2)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    shape = santa.make_shape(2, 8, 2, 128, 512)
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.empty(2, 8, 128, device=DEV)
    idx = torch.empty(2, 8, 16, dtype=torch.int32, device=DEV)
    assert santa.device_status(None) == 0
    bad = torch.tensor([513, 300], dtype=torch.int32, device=DEV)
    good = torch.tensor([512, 300], dtype=torch.int32, device=DEV)
    assert _call_static(lib, shape, qd, kd, vd, bad, 16, santa.SYSTEMATIC, 1, out, idx, stream) == 0
    # a later valid call on the same stream leaves the word as it is
    assert _call_static(lib, shape, qd, kd, vd, good, 16, santa.SYSTEMATIC, 1, out, idx, stream) == 0
    assert santa.device_status(None) & santa.DEV_BAD_SEQLEN
    assert santa.device_status(None) == 0  # cleared by the read
    assert _call_static(lib, shape, qd, kd, vd, bad, 16, santa.SYSTEMATIC, 1, out, idx, stream) == 0
    torch.cuda.synchronize()
    assert torch.all(idx[0] == -1) and torch.all(out[0] == 0)
    assert santa.device_status(None) & santa.DEV_BAD_SEQLEN


def test_static_scratch_rejects_oversized_problems_before_any_launch():
    lib = santa.load()
    # a workspace larger than the static buffer: refused on the host with its own status
    shape = santa.make_shape(4, 32, 8, 128, 65536)
    assert santa.workspace_size(shape, 256, santa.SYSTEMATIC) > santa.STATIC_SCRATCH_BYTES
    rc = lib.santa_decode_static(ctypes.byref(shape), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                 ctypes.c_void_p(16), ctypes.c_void_p(16), 256, santa.SYSTEMATIC,
                                 ctypes.c_uint64(0), ctypes.c_void_p(16), ctypes.c_void_p(0), ctypes.c_void_p(0))
    assert rc == santa.ERR_SCRATCH
    assert "static" in santa.status_string(rc)
