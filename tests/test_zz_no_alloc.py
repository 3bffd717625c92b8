"""santa_decode_static: the decode entry point for callers that cannot allocate device
memory (the library supplies the scratch from a fixed device array of
SANTA_STATIC_SCRATCH_BYTES).  Checked through the C ABI against santa_decode with a
caller-owned workspace, on two calls in a row, in every mode.

The file name makes pytest collect it last, so that a run stopping at the first failure
has already run every other test.  It also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from stochastic_sparse_kv_gb300 import santa, workloads
from tests.parity_util import EST_TOL

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


@pytest.mark.parametrize("mode", [santa.SYSTEMATIC, santa.STRATIFIED, santa.IID, santa.DENSE,
                                  santa.SYSTEMATIC | santa.GROUP_DEDUP])
def test_static_scratch_matches_workspace_entry_point(mode):
    lib = santa.load()
    seq = [3000, 777, 0, 2049]
    w, q, k, v, sl = workloads.small("static", len(seq), 16, 4, 128, 3000, 96, seq_lens=seq, seed=21)
    qd, kd, vd, sld = q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)
    B, H_q, d = q.shape
    S = 96
    shape = santa.make_shape(B, H_q, 4, d, 3000)
    stream = torch.cuda.current_stream().cuda_stream
    ws = santa.new_workspace(santa.workspace_size(shape, S, mode), DEV)
    sampled = (mode & 0xff) != santa.DENSE
    for seed in (5, 6):  # two calls in a row, each against the workspace entry point
        out_a = torch.full((B, H_q, d), float("nan"), device=DEV)
        out_b = torch.full((B, H_q, d), float("nan"), device=DEV)
        idx_a = torch.full((B, H_q, S), -7, dtype=torch.int32, device=DEV) if sampled else None
        idx_b = torch.full((B, H_q, S), -7, dtype=torch.int32, device=DEV) if sampled else None
        assert _call_static(lib, shape, qd, kd, vd, sld, S, mode, seed, out_a, idx_a, stream) == 0
        assert _call_workspace(lib, shape, qd, kd, vd, sld, S, mode, seed, out_b, idx_b, ws, stream) == 0
        torch.cuda.synchronize()
        oa, ob = out_a.cpu().numpy(), out_b.cpu().numpy()
        assert np.isfinite(oa).all()
        assert np.abs(oa - ob).max() <= EST_TOL
        if sampled:
            assert np.array_equal(idx_a.cpu().numpy(), idx_b.cpu().numpy())


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
