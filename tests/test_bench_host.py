"""bench.py's host-side arithmetic, checked without a GPU.

Algorithmic bytes of a decode step: all of K once, the S gathered V rows per query head,
q, the fp32 output and seq_lens; the dense path reads all of K and V.  At the
Llama-shaped batch (B=16, H_q=32, H_kv=8, d=128, 32768 keys) these are fixed numbers:
1107.7 MB at S=256 (1082.5 / 1090.9 / 1141.2 MB at S=64 / 128 / 512) and 2147.9 MB dense.
"""
import bench

SEQ = [32768] * 16


def test_algorithmic_bytes_of_the_llama_shaped_batch():
    assert bench.algorithmic_bytes(16, 32, 8, 128, SEQ, 256, "systematic") == 1107689536
    assert bench.algorithmic_bytes(16, 32, 8, 128, SEQ, 256, "stratified") == 1107689536
    assert bench.algorithmic_bytes(16, 32, 8, 128, SEQ, 256, "dense") == 2147876928
    sweep = {64: 1082.5, 128: 1090.9, 512: 1141.2}
    for S, mb in sweep.items():
        assert round(bench.algorithmic_bytes(16, 32, 8, 128, SEQ, S, "systematic") / 1e6, 1) == mb


def test_empty_rows_read_no_keys_and_gather_no_rows():
    full = bench.algorithmic_bytes(2, 32, 8, 128, [4096, 4096], 256, "systematic")
    half = bench.algorithmic_bytes(2, 32, 8, 128, [4096, 0], 256, "systematic")
    k_row_b = 8 * 4096 * 128 * 2
    v_rows_b = 32 * 256 * 128 * 2
    assert full - half == k_row_b + v_rows_b


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on():
    v = bench.profiled_traffic()
    rec = {}
    with open(bench.PROFILE_TRAFFIC) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                a, b = line.split("=", 1)
                rec[a.strip()] = b.strip()
    if rec.get("source_sha") == bench.sources_sha():
        assert v == float(rec["traffic_bytes_per_launch"]) and v > 0
    else:
        assert v is None


def test_traffic_record_key_covers_every_kernel_source():
    # a change to any kernel source, dispatch table or host launch code invalidates it
    import os
    csrc = os.path.join(bench.ROOT, bench.CSRC)
    files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    assert sorted(os.path.basename(s) for s in bench.KERNEL_SOURCES) == files
