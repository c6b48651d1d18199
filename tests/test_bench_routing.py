"""The kernel name bench.py writes into a decode line's roofline mirrors the C
ABI's routing of paged_decode_attention_multi: q_len 1 -> the decode kernel;
16-bit caches with head dim 128 and up to 32 query rows per kv head -> the
transposed tensor-core kernel; 33-64 rows -> the 128-row prefill kernel when
its grid fills the SMs, else the transposed kernel; fp8 / f32 caches, a fixed
split count or small grids of wider rows -> the decode kernel's units (8 rows;
16 on fp8 caches past 8 rows); fp8 caches -> the units too (the transposed
kernel, which widens fp8 tiles to f16, only when forced); a route forced
through pkv_set_route applies where it can.  Host logic only."""
from types import SimpleNamespace

import pytest

import bench

SMS = 152


def _w(q_len, B=64, Hq=64, Hkv=8, D=128, dtype="bf16"):
    return SimpleNamespace(q_len=q_len, B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype)


def _route(name):
    if name.startswith("mq_decode_kernel"):
        return "transposed"
    if name.startswith("prefill"):
        return "prefill"
    if "-row units" in name:
        return "units"
    return "decode"


@pytest.mark.parametrize("w,splits,want", [
    (_w(1), 0, "decode"),
    (_w(2), 0, "transposed"),                       # 16 rows
    (_w(4), 0, "transposed"),                       # 32 rows
    (_w(8), 0, "prefill"),                          # 64 rows, 512 items fill 152 SMs
    (_w(8, B=4), 0, "transposed"),                  # 64 rows, 32 items: the prefill grid would not fill
    (_w(16, Hq=64, Hkv=8), 0, "prefill"),           # 128 rows: past the transposed kernel
    (_w(16, B=4), 0, "units"),                      # 128 rows, small grid
    (_w(4, dtype="fp8_e4m3"), 0, "units"),           # fp8, 32 rows: two 16-row units
    (_w(4, dtype="fp8_e4m3", Hq=32), 0, "units"),     # the 32K fp8 layer's group 4 at q_len 4: one 16-row unit
    (_w(8, dtype="fp8_e4m3", Hq=32), 0, "units"),     # 32 rows
    (_w(8, dtype="fp8_e4m3"), 0, "units"),            # fp8, 64 rows: no fp8 prefill route
    (_w(4, dtype="f32"), 0, "units"),
    (_w(4), 7, "units"),                            # a fixed split count
    (_w(4, D=64), 0, "prefill"),                    # head dim 64: the prefill kernel
    (_w(4, D=64, B=2), 0, "units"),
    (_w(4, dtype="f16"), 0, "transposed"),
    (_w(4, B=4096), 0, "prefill"),                  # past the transposed kernel's batch bound
], ids=lambda v: str(v) if not isinstance(v, SimpleNamespace) else f"L{v.q_len}-B{v.B}-D{v.D}-{v.dtype}")
def test_roofline_kernel_follows_the_routing(w, splits, want):
    assert _route(bench.attention_kernel_name(w, splits, SMS)) == want


@pytest.mark.parametrize("w,rows", [
    (_w(4, dtype="fp8_e4m3", Hq=32), 16),           # 16 rows per kv head
    (_w(8, dtype="fp8_e4m3"), 16),                  # 64 rows: four 16-row units
    (_w(1, dtype="fp8_e4m3", Hq=8, Hkv=1), 8),      # q_len 1 takes the plain decode name
    (_w(4, dtype="f32"), 8),
    (_w(4, D=64, B=2), 8),
], ids=lambda v: str(v) if not isinstance(v, SimpleNamespace) else f"L{v.q_len}-{v.dtype}-q{v.Hq}")
def test_unit_width_in_the_kernel_name(w, rows):
    name = bench.attention_kernel_name(w, 0, SMS, force="units")
    if w.q_len == 1:
        assert "units" not in name
    else:
        assert f"{rows}-row units" in name


@pytest.mark.parametrize("force,w,want", [
    ("prefill", _w(4), "prefill"),
    ("units", _w(4), "units"),
    ("transposed", _w(8), "transposed"),            # forced on 64 rows with a full prefill grid
    ("transposed", _w(16), "prefill"),              # cannot apply past 64 rows
    ("transposed", _w(4, dtype="fp8_e4m3", Hq=32), "transposed"),  # fp8 at 16 rows, forced
])
def test_roofline_kernel_honours_the_override(force, w, want):
    assert _route(bench.attention_kernel_name(w, 0, SMS, force)) == want
