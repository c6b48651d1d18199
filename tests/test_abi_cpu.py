"""CPU checks of the C ABI: the library loads, exports every function that
include/pagedkv.h declares, and rejects invalid arguments before touching a
GPU.  No compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_03_gb300 as pkv
    return pkv


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(p(?:aged|kv)_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    pkv = _lib()
    names = _declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(pkv.lib(), n), n


def test_status_strings_and_version():
    pkv = _lib()
    assert pkv.pkv_version() >= 10000
    for code in range(-8, 1):
        assert pkv.pkv_status_string(code) != "unknown status"


NULL = None


def _attn(L, **kw):
    a = dict(out=16, q=16, q_dtype=2, k=16, v=16, cdt=2, ks=NULL, vs=NULL, bt=16, mb=4, cl=16,
             B=2, Hq=8, Hkv=2, D=128, nb=10, scale=0.1, ns=3, ws=256, wsb=1 << 30, stream=NULL)
    a.update(kw)
    return L.paged_decode_attention(a["out"], a["q"], a["q_dtype"], a["k"], a["v"], a["cdt"],
                                    a["ks"], a["vs"], a["bt"], a["mb"], a["cl"], a["B"], a["Hq"],
                                    a["Hkv"], a["D"], a["nb"], a["scale"], a["ns"], a["ws"],
                                    a["wsb"], a["stream"])


def test_decode_argument_errors_without_gpu():
    pkv = _lib()
    L = pkv.lib()
    assert _attn(L, Hq=6, Hkv=4) == pkv.PKV_EINVAL          # Hq % Hkv != 0
    assert _attn(L, D=96) == pkv.PKV_EUNSUPPORTED             # head dim
    assert _attn(L, q_dtype=1) == pkv.PKV_EUNSUPPORTED        # q must match a bf16 cache
    assert _attn(L, cdt=0, q_dtype=2) == pkv.PKV_EUNSUPPORTED  # fp32 cache needs fp32 q
    assert _attn(L, q_dtype=3, cdt=3) == pkv.PKV_EINVAL       # fp8 queries
    assert _attn(L, cdt=9) == pkv.PKV_EINVAL
    assert _attn(L, out=NULL) == pkv.PKV_EINVAL
    assert _attn(L, bt=NULL) == pkv.PKV_EINVAL
    assert _attn(L, cdt=3, ks=16, vs=NULL) == pkv.PKV_EINVAL   # fp8 needs both scales
    assert _attn(L, q=18) == pkv.PKV_EINVAL                   # misaligned
    assert _attn(L, scale=float("nan")) == pkv.PKV_EINVAL
    assert _attn(L, nb=0) == pkv.PKV_EINVAL
    assert _attn(L, ns=-1) == pkv.PKV_EINVAL
    assert _attn(L, ws=NULL) == pkv.PKV_EWORKSPACE
    assert _attn(L, ws=128) == pkv.PKV_EWORKSPACE             # not 256-aligned
    assert _attn(L, wsb=64) == pkv.PKV_EWORKSPACE             # too small
    assert _attn(L, B=0) == pkv.PKV_OK                        # nothing to do


def test_multi_query_argument_errors_without_gpu():
    pkv = _lib()
    L = pkv.lib()

    def multi(q_len, **kw):
        a = dict(B=2, Hq=8, Hkv=2, D=128, ws=256, wsb=1 << 30)
        a.update(kw)
        return L.paged_decode_attention_multi(16, 16, 2, 16, 16, 2, NULL, NULL, 16, 4, 16, a["B"],
                                              q_len, a.get("window", 0), a["Hq"], a["Hkv"], a["D"],
                                              10, 0.1, 3, a["ws"], a["wsb"], NULL)
    assert multi(0) == pkv.PKV_EINVAL
    assert multi(65) == pkv.PKV_EINVAL                        # above PKV_MAX_Q_LEN
    assert multi(4, Hq=6, Hkv=4) == pkv.PKV_EINVAL
    assert multi(4, ws=NULL) == pkv.PKV_EWORKSPACE
    assert multi(4, window=-1) == pkv.PKV_EINVAL
    assert multi(4, B=0) == pkv.PKV_OK
    size = ctypes.c_size_t(0)
    assert L.paged_decode_multi_workspace_bytes(2, 0, 8, 2, 128, 2, 2, 5, ctypes.byref(size)) == pkv.PKV_EINVAL
    assert L.paged_decode_multi_workspace_bytes(2, 4, 8, 2, 128, 2, 2, 5, ctypes.byref(size)) == pkv.PKV_OK
    one = ctypes.c_size_t(0)
    assert L.paged_decode_workspace_bytes(2, 8, 2, 128, 2, 2, 5, ctypes.byref(one)) == pkv.PKV_OK
    assert size.value == one.value          # partials are per worker, not per query row


def test_workspace_grows_by_the_unit_width_per_partition():
    """Per partition the workspace holds a partial O and a log-sum-exp per
    query row of a unit and both column groups, a plan entry and a flag.
    FP8 caches with more than 8 query rows per kv head use 16-row units, so
    their partitions are twice as wide; 16-bit caches keep 8-row units."""
    pkv = _lib()
    L = pkv.lib()

    def ws(Hq, Hkv, D, cache, q, splits):
        size = ctypes.c_size_t(0)
        assert L.paged_decode_workspace_bytes(3, Hq, Hkv, D, cache, q, splits, ctypes.byref(size)) == pkv.PKV_OK
        return size.value

    def per_partition(rows, D):
        return 2 * rows * D * 4 + 2 * rows * 4 + 16 + 4

    BF16, FP8 = 2, 3  # PKV_BF16, PKV_FP8_E4M3 in include/pagedkv.h
    for Hq, Hkv, D, cache, rows in [(32, 2, 128, FP8, 16), (32, 2, 64, FP8, 16), (16, 2, 128, FP8, 8),
                                    (32, 2, 128, BF16, 8), (64, 8, 128, BF16, 8)]:
        # 256 partitions more: every region grows by a multiple of its 256-byte alignment
        assert ws(Hq, Hkv, D, cache, BF16, 1280) - ws(Hq, Hkv, D, cache, BF16, 1024) == 256 * per_partition(rows, D)
    # the fixed scratch of the static entry: ~1000 16-row partitions at D = 128
    cap = pkv.PKV_STATIC_SCRATCH_BYTES
    assert ws(32, 2, 128, FP8, BF16, 1000) <= cap < ws(32, 2, 128, FP8, BF16, 1100)


def test_append_copy_merge_argument_errors_without_gpu():
    pkv = _lib()
    L = pkv.lib()
    ok = dict(kn=16, vn=16, ndt=2, kc=16, vc=16, cdt=2, ks=NULL, vs=NULL, sm=16, B=2, Hkv=2, D=128, nb=4)

    def app(**kw):
        a = dict(ok); a.update(kw)
        return L.paged_kv_append(a["kn"], a["vn"], a["ndt"], a["kc"], a["vc"], a["cdt"], a["ks"],
                                 a["vs"], a["sm"], a["B"], a["Hkv"], a["D"], a["nb"], NULL)
    assert app(ndt=1) == pkv.PKV_EUNSUPPORTED      # bit-exact copy needs equal dtypes
    assert app(cdt=3) == pkv.PKV_EINVAL            # fp8 without scales
    assert app(cdt=3, ndt=3, ks=16, vs=16) == pkv.PKV_EUNSUPPORTED
    assert app(sm=NULL) == pkv.PKV_EINVAL
    assert app(D=80) == pkv.PKV_EUNSUPPORTED
    assert app(kc=8) == pkv.PKV_EINVAL
    assert app(B=0) == pkv.PKV_OK
    assert L.paged_kv_copy_blocks(16, 16, 2, NULL, NULL, NULL, 3, 2, 128, 4, NULL) == pkv.PKV_EINVAL
    assert L.paged_kv_copy_blocks(16, 16, 3, NULL, NULL, 16, 3, 2, 128, 4, NULL) == pkv.PKV_EINVAL
    assert L.paged_kv_copy_blocks(16, 16, 2, NULL, NULL, 16, 0, 2, 128, 4, NULL) == pkv.PKV_OK
    assert L.paged_decode_merge(16, 2, 16, 16, 2, 4, 128, 0, NULL) == pkv.PKV_EINVAL
    assert L.paged_decode_merge(16, 3, 16, 16, 2, 4, 128, 2, NULL) == pkv.PKV_EINVAL
    assert L.paged_decode_merge(NULL, 2, 16, 16, 2, 4, 128, 2, NULL) == pkv.PKV_EINVAL
    size = ctypes.c_size_t(0)
    assert L.paged_decode_workspace_bytes(2, 8, 3, 128, 2, 2, 0, ctypes.byref(size)) == pkv.PKV_EINVAL
    assert L.paged_decode_workspace_bytes(2, 8, 2, 128, 2, 2, 5, ctypes.byref(size)) == pkv.PKV_OK
    assert size.value > 5 * 2 * 8 * 128 * 4


def test_import_fails_loudly_without_library(tmp_path):
    """The binding refuses to import when the shared library is absent."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "paged_kv_gqa_03_gb300"
    shutil.copytree(os.path.join(ROOT, "paged_kv_gqa_03_gb300"), pkg,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import paged_kv_gqa_03_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "ImportError" in r.stderr
