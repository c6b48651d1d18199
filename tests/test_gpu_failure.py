"""The timeout path of the kernels' bounded waits, made to happen without a
fault or a hang.  pkv_test_stall_next limits every wait of the next call to
a few milliseconds and makes one consumer wait on a barrier nothing
completes; that wait gives up, the kernel flags PKV_FLAG_TIMEOUT, lets its
copies (and tensor-core operations) in flight complete, frees its tensor
memory and exits.  The checks: the call's status reports the timeout within
a bound of a fraction of a second, and the next ordinary call on the same
workspace (decode) or status word (prefill) is clean and matches the oracle.
No wait in any of this is unbounded."""
import math
import time

import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import compare, routes, run_gpu_step, run_oracle_step

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000      # 20 ms per wait in the stalled call


def _pkv():
    import paged_kv_gqa_03_gb300 as pkv
    return pkv


@pytest.mark.parametrize("cfg,spec", [
    (3, dict(B=4, ctx=[300, 41, 1000, 17], free_frac=0.3, min_free=4)),   # bf16, group 8
    (5, dict(B=2, ctx=[700, 40], free_frac=0.3, min_free=2)),              # fp8, group 4
])
def test_decode_wait_runs_out_and_the_next_call_is_exact(cfg, spec):
    pkv = _pkv()
    w = workloads.config(cfg, **spec)
    step, out = run_gpu_step(w)
    *_, ref = run_oracle_step(w)
    compare(out, ref, w.dtype, "before the stall")
    q = w.q.to("cuda")

    pkv.pkv_test_stall_next("decode", LIMIT_NS)
    stalled = torch.zeros_like(out)
    t0 = time.perf_counter()
    step.attend(q, stalled)
    rc, flags = pkv.paged_decode_status(step.workspace, step.stream)
    dt = time.perf_counter() - t0
    assert rc == pkv.PKV_ETIMEOUT and flags & pkv.PKV_FLAG_TIMEOUT, (rc, flags)
    assert dt < 2.0, f"the stalled call took {dt:.2f} s"

    again = torch.full_like(out, float("nan"))
    step.attend(q, again)
    rc, flags = pkv.paged_decode_status(step.workspace, step.stream)
    assert (rc, flags) == (pkv.PKV_OK, 0)
    compare(again, ref, w.dtype, "the call after the stall")


def test_stall_request_is_one_shot_and_validated():
    pkv = _pkv()
    with pytest.raises(pkv.PagedKVError):
        pkv.pkv_test_stall_next("decode", 10)              # below 1 ms
    with pytest.raises(pkv.PagedKVError):
        pkv.pkv_test_stall_next("decode", 20_000_000_000)  # above 10 s
    pkv.pkv_test_stall_next("decode", LIMIT_NS)
    pkv.pkv_test_stall_next("decode", 0)                   # cancelled: the next call is ordinary
    w = workloads.config(3, B=2, ctx=[100, 33], free_frac=0.3, min_free=2)
    step, out = run_gpu_step(w)
    rc, flags = pkv.paged_decode_status(step.workspace, step.stream)
    assert (rc, flags) == (pkv.PKV_OK, 0)
    *_, ref = run_oracle_step(w)
    compare(out, ref, w.dtype, "after a cancelled request")


@pytest.mark.parametrize("kernel", ["persistent", "tiles"])
def test_prefill_wait_runs_out_and_the_next_call_is_exact(kernel):
    pkv = _pkv()
    import oracle
    c = workloads.make_prefill(7, n=[130, 5, 257], prefix=[1000, 33, 16], Hq=16, Hkv=2, D=128, dtype="bf16")
    dev = "cuda"
    q = c["q"].to(dev)
    kc, vc = c["kc"].to(dev), c["vc"].to(dev)
    table = torch.from_numpy(c["table"]).to(dev)
    lens = torch.from_numpy(c["ctx"]).to(dev)
    q_start = torch.from_numpy(c["q_start"]).to(dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(c["D"])

    def call(out):
        pkv.paged_prefill_attention(out, q, kc, vc, table, lens, q_start, max(c["n"]), scale, status=status)
        torch.cuda.synchronize()
        return int(status.item())

    with routes(prefill=kernel):
        pkv.pkv_test_stall_next("prefill", LIMIT_NS)
        t0 = time.perf_counter()
        flags = call(torch.zeros_like(q))
        dt = time.perf_counter() - t0
        assert flags & pkv.PKV_FLAG_TIMEOUT, flags
        assert dt < 2.0, f"the stalled call took {dt:.2f} s"
        out = torch.full_like(q, float("nan"))
        assert call(out) == 0
    ref = oracle.prefill(c["q"], "bf16", c["kc"], c["vc"], "bf16", c["table"], c["ctx"], c["q_start"], scale=scale)
    compare(out, ref, "bf16", f"prefill ({kernel}) after the stall")
    assert np.isfinite(ref).all()
