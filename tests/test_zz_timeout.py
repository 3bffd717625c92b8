"""The kernels' bounded waits.  With a very short limit (santa_set_wait_limit) a decode
call's pipeline waits run out: the kernels report SANTA_DEV_TIMEOUT through the device
error word, drain their asynchronous copies and MMAs, and exit, and the context stays
usable -- the next call with the default limit reproduces the reference result.  No GPU
fault or hang is involved: the waits simply give up early.

The file name makes pytest collect it after the other GPU tests.
"""
import pytest
import torch

from stochastic_sparse_kv_gb300 import santa, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("mode,B,two_pass", [("systematic", 4, True), ("dense", 4, False), ("systematic", 1, False)])
def test_short_wait_limit_reports_a_timeout_and_leaves_the_context_usable(mode, B, two_pass):
    """(two_pass: the score and value stages as two launches; B=1: the single-pass cluster
    kernel, whose CTAs all still reach every cluster barrier after their waits give up)"""
    seq = [16384, 16384, 9000, 16384][:B]
    _, q, k, v, sl = workloads.small("timeout", B, 32, 8, 128, 16384, 256, seq_lens=seq, seed=31)
    qd, kd, vd, sld = q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)
    shape = santa.make_shape(B, 32, 8, 128, 16384)
    assert santa.call_info(shape, 256, mode, two_pass=two_pass) == (1 if B == 1 else 2)
    ws = santa.new_workspace(santa.workspace_size(shape, 256, mode), DEV)
    ref, iref = santa.decode(qd, kd, vd, sld, 256, mode, seed=3, workspace=ws, two_pass=two_pass)
    ref = ref.clone()
    iref = iref.clone() if iref is not None else None
    torch.cuda.synchronize()
    assert santa.device_status(ws) == 0
    try:
        santa.set_wait_limit(1)  # 1 ns: the first wait that is not already satisfied gives up
        santa.decode(qd, kd, vd, sld, 256, mode, seed=3, workspace=ws, two_pass=two_pass)
        torch.cuda.synchronize()
        code = santa.device_status(ws)
    finally:
        santa.set_wait_limit(0)
    assert code & santa.DEV_TIMEOUT
    assert santa.device_status(ws) == 0  # cleared by the read
    out, idx = santa.decode(qd, kd, vd, sld, 256, mode, seed=3, workspace=ws, two_pass=two_pass)
    torch.cuda.synchronize()
    assert santa.device_status(ws) == 0
    assert torch.equal(out, ref)
    if mode != "dense":
        assert torch.equal(idx, iref)
