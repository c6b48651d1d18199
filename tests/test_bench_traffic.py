"""bench.py's roofline `traffic` comes from a committed ncu record of the
dominant kernel: DRAM reads scaled by the K/V bytes the launch attends,
writes as captured.  A record is used only for its own q_len and only while
the hash of the kernel's sources matches the one it was captured with.
Host logic only."""
import hashlib
import json
import os
from types import SimpleNamespace

import bench


def _w(q_len=1, dtype="fp8_e4m3", kv=1000):
    return SimpleNamespace(q_len=q_len, dtype=dtype, window=0, prefix_blocks=0, kv_bytes=lambda: kv)


def _record(tmp, name, q_len, good=True, sources=("common.cuh", "decode.cuh", "internal.h")):
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(bench.ROOT, "paged_kv_gqa_03_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    rec = {"kv_bytes": 500, "dram_bytes_read": 510, "dram_bytes_write": 7, "q_len": q_len,
           "sources": list(sources), "source_sha256": h.hexdigest() if good else "0" * 64}
    with open(os.path.join(tmp, name), "w") as f:
        json.dump(rec, f)


def test_record_scaled_by_the_attended_bytes(tmp_path):
    _record(tmp_path, "decode_traffic_fp8.json", 1)
    assert bench.kernel_traffic(_w(kv=1000), profiles_dir=str(tmp_path)) == int(510 / 500 * 1000 + 7)


def test_record_for_another_q_len_or_stale_sources_is_not_used(tmp_path):
    _record(tmp_path, "decode_traffic_fp8.json", 1)
    assert bench.kernel_traffic(_w(q_len=4), profiles_dir=str(tmp_path)) is None
    _record(tmp_path, "decode_traffic_fp8_qlen4.json", 4, good=False)
    assert bench.kernel_traffic(_w(q_len=4), profiles_dir=str(tmp_path)) is None
    _record(tmp_path, "decode_traffic_fp8_qlen4.json", 4)
    assert bench.kernel_traffic(_w(q_len=4, kv=2000), profiles_dir=str(tmp_path)) == int(510 / 500 * 2000 + 7)


def test_shared_prefix_and_window_workloads_have_no_record(tmp_path):
    _record(tmp_path, "decode_traffic.json", 1)
    w = _w(dtype="bf16")
    w.prefix_blocks = 24
    assert bench.kernel_traffic(w, profiles_dir=str(tmp_path)) is None
    w = _w(dtype="bf16")
    w.window = 1024
    assert bench.kernel_traffic(w, profiles_dir=str(tmp_path)) is None
    assert bench.kernel_traffic(_w(dtype="bf16"), profiles_dir=str(tmp_path)) is not None
