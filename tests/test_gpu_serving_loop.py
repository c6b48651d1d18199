"""A decode serving loop through the public API (DecodeStep.run): each step
copies its inputs and bookkeeping from pinned host memory, appends and
attends through one captured graph per staging buffer, and writes the output
into pinned host memory, while the host prepares the next step's slot
mapping.  Contexts advance one token per sequence per step, blocks open
every 16 tokens, and the first step copies a block shared with a fork
(copy-on-write, run eagerly).  Every step's output and the final caches
against the oracle replaying the same block-table operations
("LLM推理优化实战" §2.2 block table and copy-on-write)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.block_table import BlockTable

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("q_len", [1, 3])
def test_serving_loop_steps_match_the_oracle(q_len):
    from paged_kv_gqa_03_gb300.step import DecodeStep
    from gpu_helpers import compare
    dev = "cuda"
    Hq, Hkv, D, nb, steps = 16, 2, 128, 64, 24
    g = torch.Generator().manual_seed(21)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    shape_q = (3, Hq, D) if q_len == 1 else (3, q_len, Hq, D)
    shape_kv = (3, Hkv, D) if q_len == 1 else (3, q_len, Hkv, D)
    q = torch.randn(shape_q, generator=g).to(torch.bfloat16)
    kn = torch.randn(shape_kv, generator=g).to(torch.bfloat16)
    vn = torch.randn(shape_kv, generator=g).to(torch.bfloat16)

    step = DecodeStep(kc.to(dev), vc.to(dev), Hq, torch.bfloat16, 16, q_len=q_len, stream=torch.cuda.Stream())
    ref = BlockTable(nb)
    for m in (step.bm, ref):
        assert m.allocate(0, 37) and m.allocate(1, 5)
        assert m.fork(0, 2)                      # sequence 2 shares 0's partial last block
    step.seqs = [0, 1, 2]
    hout = torch.empty(shape_q, dtype=torch.bfloat16).pin_memory()
    kr, vr = kc.clone(), vc.clone()
    step.prepare()
    step.stage_inputs(q, kn, vn, both=True)
    cows = 0
    for n in range(steps):
        slots, cow = ref.append_slots([s for s in (0, 1, 2) for _ in range(q_len)])
        assert step.h_slots.tolist() == slots
        cows += len(cow)
        step.run(hout)
        table = np.asarray(step.h_table).copy()
        lens = np.asarray(step.h_lens).copy()
        if n + 1 < steps:
            step.prepare()                       # the next step's a1 while this one runs
        step.stream.synchronize()
        for src, dst in cow:
            kr[dst], vr[dst] = kr[src], vr[src]
        kr, vr, _, _ = oracle.append(kr, vr, "bf16", kn.reshape(-1, Hkv, D), vn.reshape(-1, Hkv, D), "bf16",
                                     slots)
        want = oracle.decode(q, "bf16", kr, vr, "bf16", table, lens, scale=1.0 / np.sqrt(D))
        compare(hout, want, "bf16", f"serving loop step {n}")
    assert cows == 1                             # the first step's write into the shared block
    assert np.array_equal(step.k_cache.cpu().view(torch.int16).numpy(), kr.view(np.int16))
    assert np.array_equal(step.v_cache.cpu().view(torch.int16).numpy(), vr.view(np.int16))


@pytest.mark.parametrize("q_len", [1, 2])
def test_serving_loop_one_step_queued_ahead(q_len):
    """The loop with one step queued ahead of the host: step n is issued
    before the host waits for step n - 1 and reads its output (two pinned
    output tensors alternate), then the host prepares step n + 1 into the
    staging buffer step n - 1 read.  Every step's output against the oracle."""
    from paged_kv_gqa_03_gb300.step import DecodeStep
    from gpu_helpers import compare
    dev = "cuda"
    Hq, Hkv, D, nb, steps = 8, 2, 128, 64, 20
    g = torch.Generator().manual_seed(22)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    shape_q = (3, Hq, D) if q_len == 1 else (3, q_len, Hq, D)
    shape_kv = (3, Hkv, D) if q_len == 1 else (3, q_len, Hkv, D)
    q = torch.randn(shape_q, generator=g).to(torch.bfloat16)
    kn = torch.randn(shape_kv, generator=g).to(torch.bfloat16)
    vn = torch.randn(shape_kv, generator=g).to(torch.bfloat16)

    step = DecodeStep(kc.to(dev), vc.to(dev), Hq, torch.bfloat16, 16, q_len=q_len, stream=torch.cuda.Stream())
    ref = BlockTable(nb)
    for m in (step.bm, ref):
        assert m.allocate(0, 30) and m.allocate(1, 16) and m.allocate(2, 1)
    step.seqs = [0, 1, 2]
    houts = [torch.empty(shape_q, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    kr, vr = kc.clone(), vc.clone()
    step.prepare()
    step.stage_inputs(q, kn, vn, both=True)
    pending = None
    for n in range(steps):
        slots, cow = ref.append_slots([s for s in (0, 1, 2) for _ in range(q_len)])
        assert cow == [] and step.h_slots.tolist() == slots
        step.run(houts[n % 2])
        done = torch.cuda.Event()
        done.record(step.stream)
        table = np.asarray(step.h_table).copy()
        lens = np.asarray(step.h_lens).copy()
        kr, vr, _, _ = oracle.append(kr, vr, "bf16", kn.reshape(-1, Hkv, D), vn.reshape(-1, Hkv, D), "bf16",
                                     slots)
        want = oracle.decode(q, "bf16", kr, vr, "bf16", table, lens, scale=1.0 / np.sqrt(D))
        if pending is not None:
            ev, out, ref_out, m = pending
            ev.synchronize()
            compare(out, ref_out, "bf16", f"queued-ahead loop step {m}")
        pending = (done, houts[n % 2], want, n)
        if n + 1 < steps:
            step.prepare()
    ev, out, ref_out, m = pending
    ev.synchronize()
    compare(out, ref_out, "bf16", f"queued-ahead loop step {m}")
    assert np.array_equal(step.k_cache.cpu().view(torch.int16).numpy(), kr.view(np.int16))
