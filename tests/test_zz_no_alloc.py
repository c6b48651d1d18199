"""paged_decode_attention_static — decode attention for callers that cannot
allocate device memory (a C host without a device allocator, a plugin whose
host framework owns all device memory, a serving loop that must not call
cudaMalloc once it runs).  It runs on a fixed scratch array the library keeps
on each GPU.

The checks, through the C ABI: two calls in a row (different shapes, so the
second reuses the scratch the first left behind) give the same outputs as the
workspace-taking entry point within the attention tolerances, and match the
oracle; the status of the shared scratch reads clean after each; a shape
whose usual partition count needs more scratch than the array holds runs on
fewer partitions; an explicit partition count beyond the fixed capacity is
refused before anything runs.  This file is named to be collected last."""
import pytest
import torch

import workloads
from gpu_helpers import compare, run_gpu_step, run_oracle_step

pytestmark = pytest.mark.gpu


def _call_static(pkv, step, q, out, num_splits=0):
    pkv.paged_decode_attention_static(out, q, step.k_cache, step.v_cache, step.d_table, step.d_lens,
                                      step.scale, step.k_scale, step.v_scale,
                                      num_splits=num_splits, stream=step.stream)


def test_static_scratch_entry_matches_workspace_entry_on_two_calls():
    import paged_kv_gqa_03_gb300 as pkv
    cases = [workloads.config(3, B=6, ctx=[900, 17, 33, 1, 2048, 300], free_frac=0.3, min_free=6),
             workloads.config(5, B=3, ctx=[1500, 40, 700], free_frac=0.3, min_free=3)]
    for w in cases:
        step, out_ws = run_gpu_step(w)          # append + workspace-taking attention
        q = w.q.to("cuda")
        out_static = torch.full_like(out_ws, float("nan"))
        _call_static(pkv, step, q, out_static)
        rc, flags = pkv.paged_decode_static_status(step.stream)
        assert (rc, flags) == (pkv.PKV_OK, 0)
        compare(out_static, out_ws.double().cpu().numpy(), w.dtype, f"static scratch vs workspace ({w.name})")
        *_, ref = run_oracle_step(w)
        compare(out_static, ref, w.dtype, f"static scratch vs oracle ({w.name})")


def test_static_scratch_shrinks_the_library_partition_count_to_fit():
    """FP8 cache, 16 query rows per kv head, D 128: 16-row partials at one
    partition per resident warp need more than the fixed scratch; with
    num_splits = 0 the entry takes fewer partitions and still runs."""
    import paged_kv_gqa_03_gb300 as pkv
    w = workloads.make(dict(B=3, Hq=32, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="bf16",
                            ctx=[900, 17, 2100], free_frac=0.3, min_free=3), 4242)
    usual = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, torch.float8_e4m3fn, torch.bfloat16)
    assert usual > 16 << 20                  # the usual count does not fit
    step, out_ws = run_gpu_step(w)
    q = w.q.to("cuda")
    out_static = torch.full_like(out_ws, float("nan"))
    _call_static(pkv, step, q, out_static)
    rc, flags = pkv.paged_decode_static_status(step.stream)
    assert (rc, flags) == (pkv.PKV_OK, 0)
    compare(out_static, out_ws.double().cpu().numpy(), w.dtype, "static scratch, fewer partitions, vs workspace")
    *_, ref = run_oracle_step(w)
    compare(out_static, ref, w.dtype, "static scratch, fewer partitions, vs oracle")


def test_static_scratch_refuses_requests_beyond_its_capacity():
    import paged_kv_gqa_03_gb300 as pkv
    w = workloads.config(3, B=2, ctx=[40, 17], free_frac=0.5, min_free=2)
    step, _ = run_gpu_step(w)
    q = w.q.to("cuda")
    out = torch.zeros_like(q)
    # 2^20 partitions need far more scratch than the 16 MiB the library keeps
    with pytest.raises(pkv.PagedKVError) as e:
        _call_static(pkv, step, q, out, num_splits=1 << 20)
    assert e.value.status == pkv.PKV_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0      # nothing ran
