"""The timeline tool: its stamp arithmetic on hand-made stamp arrays (CPU), the normal
library's refusal of a stamp buffer, and one stamped run on the GPU in its own process."""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from stochastic_sparse_kv_gb300 import santa, timeline

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _two_pass_stamps():
    st = np.zeros((timeline.ROWS_SCORE + 4, 16), dtype=np.uint64)
    base = 10 ** 15
    for c in range(3):  # three score CTAs
        st[c, :4] = [base + c * 100, base + 5000 + c, base + 6000 + c, base + 7000 + c]
    for j in range(4):  # four value CTAs; the last one has no keys (entry stamp only)
        row = timeline.ROWS_SCORE + j
        st[row, 0] = base + 6500 + j * 1000
        if j < 3:
            st[row, 1:11] = base + 8000 + np.arange(1, 11) * (j + 1) * 100
    return st, base


def test_analyse_two_pass_layout():
    st, base = _two_pass_stamps()
    r = timeline.analyse(st, single_pass=False)
    assert r["ctas"] == 3 and r["value_ctas"] == 4
    assert r["marks"]["producer done"] == {"min": 5.0, "med": 5.001, "max": 5.002}
    assert r["marks"]["cta end"]["max"] == pytest.approx(7.002)
    # value CTA 0 entered at 6.5 us, before the last score CTA ended at 7.002 us
    assert r["value_ctas_entered_before_score_end"] == 1
    # phase k of value CTA j lasts (j + 1) * 0.1 us: medians over the three CTAs with keys
    for name, _, _ in timeline.VALUE_PHASES:
        assert r["phases"][name] == {"med": pytest.approx(0.2), "p90": pytest.approx(0.28), "max": pytest.approx(0.3)}
    assert r["value_total"]["max"] == pytest.approx(2.7)
    assert r["end"] == pytest.approx((8000 + 10 * 300) / 1e3)


def test_analyse_single_pass_layout():
    st = np.zeros((timeline.ROWS_SCORE, 16), dtype=np.uint64)
    for c in range(2):
        st[c, :12] = 5 * 10 ** 14 + c * 10 + np.arange(12) * 1000
    r = timeline.analyse(st, single_pass=True)
    assert r["ctas"] == 2
    assert r["marks"]["setup done"]["min"] == pytest.approx(1.0)
    assert r["end"] == pytest.approx(11.01)
    for name, _, _ in timeline.CLUSTER_PHASES:
        assert r["phases"][name]["med"] == pytest.approx(1.0)


def test_analyse_refuses_an_empty_buffer():
    with pytest.raises(ValueError):
        timeline.analyse(np.zeros((timeline.ROWS_SCORE + 1, 16), dtype=np.uint64), single_pass=False)


def test_median_over_calls():
    rs = [{"a": {"x": 1.0, "y": None}}, {"a": {"x": 3.0, "y": None}}, {"a": {"x": 2.0, "y": None}}]
    assert timeline._median_over_calls(rs) == {"a": {"x": 2.0, "y": None}}


def test_normal_build_has_no_stamps():
    lib = santa.load()
    assert lib.santa_timeline_buffer(None, 0) == -4
    assert lib.santa_timeline_buffer(ctypes.c_void_p(1 << 20), 1 << 20) == -4


@pytest.mark.gpu
@pytest.mark.parametrize("two_pass", [False, True])
def test_stamped_run_on_the_gpu(two_pass):
    # its own process: the stamped build and libsanta.so do not share one
    cmd = [sys.executable, "-m", "stochastic_sparse_kv_gb300.timeline", "--workload", "llama8b_b1_32k",
           "--calls", "3", "--warmup", "2", "--json"] + (["--two-pass"] if two_pass else [])
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    r = json.loads(out.stdout.strip().splitlines()[-1])
    assert r["layout"] == ("two launches" if two_pass else "single-pass cluster kernel")
    m = r["marks"]
    assert 0 <= m["producer done"]["min"] <= m["producer done"]["max"] <= r["end"] <= r["event_us"] + 5
    assert all(v["med"] is not None and v["med"] >= 0 for v in r["phases"].values())
    if two_pass:
        assert r["value_ctas"] == 32 and r["value_wait_done"]["min"] >= m["cta end"]["min"]
    else:
        assert r["ctas"] >= 8


def test_stamped_build_compiles_and_takes_a_buffer():
    # the stamped library (not part of build()) must keep compiling; its setter only
    # records the pointer, so it runs without a GPU
    import shutil
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not found")
    from stochastic_sparse_kv_gb300 import _build
    lib = ctypes.CDLL(_build.build(timeline=True))
    lib.santa_timeline_buffer.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    buf = ctypes.create_string_buffer(16 * 8 * (timeline.ROWS_SCORE + 64))
    assert lib.santa_timeline_buffer(ctypes.addressof(buf), len(buf)) == 0
    assert lib.santa_timeline_buffer(ctypes.addressof(buf), 16) == -1        # too small
    assert lib.santa_timeline_buffer(ctypes.addressof(buf) + 4, len(buf) - 8) == -2  # misaligned
    assert lib.santa_timeline_buffer(None, 0) == 0
