"""GPU parity of paged prefill (tcgen05 tensor cores): each sequence's new
tokens attend causally over its paged cache — the prompt itself and any
cached prefix ("LLM推理优化实战" §3.2 flash_attention; causal mask of
"苦猿的大模型日记 Day45" PART 04) — through the C ABI, against the oracle on
the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import compare
from workloads import make_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["persistent", "tiles"])
def prefill_kernel(request):
    """Every test runs on both prefill kernels (one persistent CTA per SM,
    one CTA per work item), through the library's route override of its
    automatic choice."""
    pkv = _pkv()
    prev = pkv.pkv_set_route("prefill", request.param)
    yield request.param
    pkv.pkv_set_route("prefill", prev)


def _pkv():
    import paged_kv_gqa_03_gb300 as pkv
    return pkv


def run_gpu(c, window=0, max_q_len=None, table=None):
    pkv = _pkv()
    dev = "cuda"
    q = c["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    tbl = torch.from_numpy(c["table"] if table is None else table).to(dev)
    pkv.paged_prefill_attention(out, q, c["kc"].to(dev), c["vc"].to(dev), tbl,
                                torch.from_numpy(c["ctx"]).to(dev), torch.from_numpy(c["q_start"]).to(dev),
                                max(c["n"]) if max_q_len is None else max_q_len,
                                1.0 / math.sqrt(c["D"]), window=window, status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def oracle_rows(c, rows, window=0):
    """The oracle on selected packed rows: token i of sequence b is a
    one-query decode over the first ctx_b - n_b + i + 1 positions."""
    q_start = c["q_start"]
    seq = np.searchsorted(q_start, rows, side="right") - 1
    lens = np.array([c["ctx"][b] - c["n"][b] + (r - q_start[b]) + 1 for r, b in zip(rows, seq)],
                    dtype=np.int32)
    return oracle.decode(c["q"][rows], c["dtype"], c["kc"], c["vc"], c["dtype"], c["table"][seq], lens,
                         scale=1.0 / math.sqrt(c["D"]), window=window)


@pytest.mark.parametrize("spec", [
    dict(n=[1, 77, 300], prefix=[0, 0, 0], Hq=16, Hkv=2, D=128, dtype="bf16"),          # whole prompts
    dict(n=[130, 5, 257], prefix=[1000, 33, 16], Hq=16, Hkv=2, D=128, dtype="bf16"),    # cached prefix
    dict(n=[64, 200], prefix=[0, 57], Hq=8, Hkv=8, D=64, dtype="f16"),                  # MHA, D 64
    dict(n=[90, 17, 1], prefix=[3, 0, 200], Hq=6, Hkv=2, D=128, dtype="f16"),           # group 3
    dict(n=[40, 129], prefix=[7, 0], Hq=16, Hkv=1, D=64, dtype="bf16"),                 # MQA group 16
    dict(n=[300], prefix=[0], Hq=4, Hkv=1, D=128, dtype="bf16", window=100),
    dict(n=[50, 200], prefix=[500, 90], Hq=8, Hkv=2, D=128, dtype="bf16", window=1),
    dict(n=[129, 3], prefix=[400, 1], Hq=8, Hkv=2, D=64, dtype="f16", window=160),
], ids=lambda s: f"{s['dtype']}-q{s['Hq']}-kv{s['Hkv']}-d{s['D']}-n{max(s['n'])}-W{s.get('window', 0)}")
def test_prefill_against_oracle(spec):
    spec = dict(spec)
    window = spec.pop("window", 0)
    c = make_prefill(7, **spec)
    out, status = run_gpu(c, window=window)
    assert status == 0
    ref = oracle.prefill(c["q"], c["dtype"], c["kc"], c["vc"], c["dtype"], c["table"], c["ctx"],
                         c["q_start"], scale=1.0 / math.sqrt(c["D"]), window=window)
    compare(out, ref, c["dtype"], "prefill")


@pytest.mark.parametrize("dtype,Hq,Hkv,D,n,prefix,window", [
    ("f16", 16, 16, 64, [2048], [0], 0),                 # the pages' prefill benchmark shape
    ("bf16", 64, 8, 128, [2048, 2048], [0, 0], 0),        # Llama-3.1-70B-shaped GQA layer
    ("bf16", 64, 8, 128, [1024, 1024], [4096, 3000], 0),  # chunked prefill after a cached prefix
    ("bf16", 64, 8, 128, [2048], [2048], 1024),           # sliding window
])
def test_prefill_large_sampled(dtype, Hq, Hkv, D, n, prefix, window):
    """Large prompts: every output finite; against the oracle, every row of
    three whole 128-row work tiles of every kv head of every sequence (the
    first, a middle and the last: token-major rows, 128 / G new tokens of all
    query heads), plus 96 rows spread over the range."""
    c = make_prefill(11, n, prefix, Hq, Hkv, D, dtype, free=8)
    out, status = run_gpu(c, window=window)
    assert status == 0
    assert torch.isfinite(out.float()).all()
    total = int(c["q_start"][-1])
    G = Hq // Hkv
    per_tile = 128 // G                      # new tokens of one 128-row tile
    tiles = []
    for b, nb in enumerate(c["n"]):
        t_last = (nb * G - 1) // 128
        for t in sorted({0, t_last // 2, t_last}):
            lo = int(c["q_start"][b]) + t * per_tile
            tiles.append(np.arange(lo, min(lo + per_tile, int(c["q_start"][b + 1]))))
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate(tiles + [[0, total - 1, 15, 16, 127, 128, total // 2],
                                             rng.choice(total, 89, replace=False)]))
    ref = oracle_rows(c, rows, window=window)
    compare(out[torch.from_numpy(rows).cuda()], ref, dtype, "prefill sampled")


def test_prefill_flags_and_empty_sequences():
    """An out-of-range block id is flagged (and read as zeros), a new-token
    count above max_q_len is flagged; sequences without new tokens are
    skipped; the other rows stay exact."""
    c = make_prefill(5, [20, 0, 33], [10, 40, 0], 8, 2, 128, "bf16")
    out, status = run_gpu(c)
    assert status == 0
    ref = oracle.prefill(c["q"], "bf16", c["kc"], c["vc"], "bf16", c["table"], c["ctx"], c["q_start"],
                         scale=1.0 / math.sqrt(128))
    compare(out, ref, "bf16", "prefill with an empty sequence")
    bad = c["table"].copy()
    bad[0, 0] = 10_000
    out, status = run_gpu(c, table=bad)
    assert status == _pkv().PKV_FLAG_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    out, status = run_gpu(c, max_q_len=20)            # sequence 2 has 33 new tokens
    assert status == _pkv().PKV_FLAG_BAD_LEN
    compare(out[:20], ref[:20], "bf16", "rows inside max_q_len")


def test_prefill_items_without_context_in_a_persistent_grid():
    """608 work items (4 sequences x 8 kv heads x 19 row tiles), so each
    persistent CTA walks several; sequence 0 keeps 300 new tokens but only
    100 positions, so its first 12 row tiles see no position and stream no
    K / V tile, interleaved with items that do.  Every output against the
    oracle, rows without context 0."""
    c = make_prefill(13, [300, 120, 250, 64], [0, 40, 7, 0], 64, 8, 128, "bf16")
    c["ctx"] = c["ctx"].copy()
    c["ctx"][0] = 100
    out, status = run_gpu(c)
    assert status == 0
    assert torch.all(out[:200].float() == 0)
    ref = oracle.prefill(c["q"], "bf16", c["kc"], c["vc"], "bf16", c["table"], c["ctx"], c["q_start"],
                         scale=1.0 / math.sqrt(128))
    compare(out, ref, "bf16", "prefill with rows without context")


@pytest.mark.parametrize("spec", [
    dict(n=[3, 1, 4, 2], prefix=[500, 37, 0, 129], Hq=16, Hkv=2, D=128, dtype="bf16"),   # <= 32 rows: 4 replicas
    dict(n=[8, 5, 1], prefix=[300, 1000, 16], Hq=8, Hkv=1, D=64, dtype="f16"),           # <= 64 rows: 2 replicas
    dict(n=[2, 1], prefix=[333, 40], Hq=16, Hkv=1, D=64, dtype="bf16"),                  # MQA group 16, 4 replicas
    dict(n=[6, 3], prefix=[2500, 200], Hq=8, Hkv=2, D=128, dtype="f16"),                 # group 4, 24 rows
    dict(n=[4, 4], prefix=[700, 50], Hq=16, Hkv=2, D=128, dtype="bf16", window=100),
    dict(n=[8, 2], prefix=[900, 5], Hq=16, Hkv=2, D=64, dtype="bf16", window=37),        # 2 replicas, window
], ids=lambda s: f"{s['dtype']}-q{s['Hq']}-kv{s['Hkv']}-d{s['D']}-n{max(s['n'])}-W{s.get('window', 0)}")
def test_prefill_few_rows_per_item(spec):
    """Items of at most 64 query rows (a few new tokens of one GQA group, the
    speculative-verify shape): the one-CTA-per-item kernel runs replicas of
    the rows over disjoint k-steps and merges them; every output against
    the oracle."""
    spec = dict(spec)
    window = spec.pop("window", 0)
    c = make_prefill(17, **spec)
    out, status = run_gpu(c, window=window)
    assert status == 0
    ref = oracle.prefill(c["q"], c["dtype"], c["kc"], c["vc"], c["dtype"], c["table"], c["ctx"],
                         c["q_start"], scale=1.0 / math.sqrt(c["D"]), window=window)
    compare(out, ref, c["dtype"], "prefill, few rows per item")


def test_prefill_few_rows_without_context():
    """Four-row items where one sequence has no context at all (its item
    streams no tile) and one sees only its first positions: zeros where
    nothing is visible, the oracle elsewhere."""
    c = make_prefill(23, [4, 4, 3], [60, 10, 0], 16, 2, 128, "bf16")
    c["ctx"] = c["ctx"].copy()
    c["ctx"][1] = 0
    c["ctx"][2] = 2
    out, status = run_gpu(c)
    assert status == 0
    assert torch.all(out[4:8].float() == 0) and torch.all(out[8].float() == 0)
    ref = oracle.prefill(c["q"], "bf16", c["kc"], c["vc"], "bf16", c["table"], c["ctx"], c["q_start"],
                         scale=1.0 / math.sqrt(128))
    compare(out, ref, "bf16", "few rows, no context")


def test_prefill_bf16_v_over_the_whole_bf16_range_is_exact():
    """V values far outside the f16 range (1e5, 3e20, -2e30) and below its
    normal range (1e-30) enter P . V as stored: every row of both sequences
    matches the oracle (the weights go in as a bf16 high part plus residual,
    V is never narrowed), and no status bit is set."""
    c = make_prefill(29, [40, 30], [100, 20], 8, 2, 128, "bf16")
    vc = c["vc"].clone()
    vc[int(c["table"][0, 2]), 1, 5, 7] = 1.0e5          # sequence 0, position 37, kv head 1
    vc[int(c["table"][0, 3]), 0, 2, 0] = 3.0e20         # sequence 0, position 50, kv head 0
    vc[int(c["table"][1, 1]), 1, 0, 100] = -2.0e30      # sequence 1, position 16, kv head 1
    vc[int(c["table"][1, 0]), 0, 3, 9] = 1.0e-30        # sequence 1, position 3, kv head 0
    out, status = run_gpu(dict(c, vc=vc))
    assert status == 0
    ref = oracle.prefill(c["q"], "bf16", c["kc"], vc, "bf16", c["table"], c["ctx"], c["q_start"],
                         scale=1.0 / math.sqrt(128))
    assert np.isfinite(ref).all()
    compare(out, ref, "bf16", "V over the bf16 range")
