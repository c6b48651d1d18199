"""paged_decode_attention_static — decode attention for callers that cannot
allocate device memory (a C host without a device allocator, a plugin whose
host framework owns all device memory, a serving loop that must not call
cudaMalloc).  It runs on a fixed scratch array the library keeps on each GPU.

The check: through the C ABI, two calls in a row (different shapes, so the
second reuses the scratch the first left behind) give the same outputs as the
workspace-taking entry point, within the attention tolerances; a request that
needs more scratch than the fixed capacity is refused before anything runs.
This file is named to be collected last."""
import ctypes

import pytest
import torch

import workloads
from gpu_helpers import compare, run_gpu_step

pytestmark = pytest.mark.gpu


def _static_fn():
    import paged_kv_gqa_03_gb300 as pkv
    fn = pkv.lib().paged_decode_attention_static
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [P, P, i32, P, P, i32, P, P, P, i32, P, i32, i32, i32, i32, i64,
                   ctypes.c_float, i32, P]
    fn.restype = i32
    return pkv, fn


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call_static(fn, pkv, step, q, out, num_splits=0):
    qd = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[q.dtype]
    cd = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2,
          torch.float8_e4m3fn: 3}[step.k_cache.dtype]
    B, Hq, D = q.shape
    return fn(_ptr(out), _ptr(q), qd, _ptr(step.k_cache), _ptr(step.v_cache), cd,
              _ptr(step.k_scale), _ptr(step.v_scale), _ptr(step.d_table), step.max_blocks,
              _ptr(step.d_lens), B, Hq, step.Hkv, D, step.num_blocks, step.scale, num_splits,
              step.stream.cuda_stream)


def test_static_scratch_entry_matches_workspace_entry_on_two_calls():
    pkv, fn = _static_fn()
    cases = [workloads.config(3, B=6, ctx=[900, 17, 33, 1, 2048, 300], free_frac=0.3, min_free=6),
             workloads.config(5, B=3, ctx=[1500, 40, 700], free_frac=0.3, min_free=3)]
    for w in cases:
        step, out_ws = run_gpu_step(w)          # append + workspace-taking attention
        q = w.q.to("cuda")
        out_static = torch.full_like(out_ws, float("nan"))
        rc = _call_static(fn, pkv, step, q, out_static)
        assert rc == 0, pkv.pkv_status_string(rc)
        step.stream.synchronize()
        ref = out_ws.double().cpu().numpy()
        compare(out_static, ref, w.dtype, f"static scratch vs workspace ({w.name})")


def test_static_scratch_refuses_requests_beyond_its_capacity():
    pkv, fn = _static_fn()
    w = workloads.config(3, B=2, ctx=[40, 17], free_frac=0.5, min_free=2)
    step, _ = run_gpu_step(w)
    q = w.q.to("cuda")
    out = torch.zeros_like(q)
    # 2^20 partitions need far more scratch than the 16 MiB the library keeps
    rc = _call_static(fn, pkv, step, q, out, num_splits=1 << 20)
    assert rc == pkv.PKV_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0      # nothing ran
