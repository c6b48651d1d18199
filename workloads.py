"""Seeded synthetic decode-step workloads.

The one module that both the CUDA path's callers (tests, bench, smoke) and
the oracle's callers draw inputs from.  It holds no arithmetic of the method:
it only draws random numbers, lays them out in the paged cache format and
writes the block tables that a block manager would adopt.

Recipe (the same for every workload):
  * torch CPU generator, seed = 1000 + workload index (explicit seeds for ad-hoc
    specs); draws in this order: context lengths, block permutation, K pool,
    V pool, q;
  * every value ~ N(0, 1) in fp32, then rounded to the storage dtype;
  * the physical block pool is a random permutation; sequence b takes the next
    ceil(cached_b / 16) blocks of it (a shared prefix takes the first blocks
    and every sequence references them);
  * every position of every block holds a random value, including positions
    past a sequence's length (stale data that attention must mask);
  * the appended token of sequence b is the value the pool already holds at
    position cached_b; that position is then zeroed, so the cache only holds
    the token after the append writes it;
  * fp8 pools: values are rounded to the new-token dtype (bf16) first, each
    (block, kv-head) tile gets scale = max|x| / 448 over its 16 positions, and
    the tile is stored as e4m3 of x / scale (torch's float8_e4m3fn cast).

`context_lens` of a workload are attended lengths, i.e. cached + 1.

A spec with `q_len` = L > 1 (several new tokens per sequence, as in the verify
step of speculative decoding) appends L tokens per sequence: `ctx` still
gives attended lengths, cached = ctx - L, q is [B, L, Hq, D] and k_new / v_new
are [B, L, Hkv, D] (token t of sequence b at position cached_b + t), each taken
from the pool and zeroed as above.  Without `q_len` the draws are unchanged.
(`q_len` = 1 given explicitly keeps the 4-D shapes with L = 1.)  A spec's
`window` (sliding window, 0 = none) changes no draw; it is carried to the
attention call and to kv_bytes.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import math
import torch

BLOCK = 16

_TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
          "fp8_e4m3": torch.float8_e4m3fn}
ITEMSIZE = {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1}

# The five decode-step workloads (1-based index = seed offset).
SPECS = {
    1: dict(name="tiny paged decode, GQA group 2, fp32, D=64",
            B=4, Hq=4, Hkv=2, D=64, dtype="f32", q_dtype="f32",
            ctx=[17, 40, 64, 100], pool=32),
    2: dict(name="Llama-2-7B-shaped MHA decode layer, fp16",
            B=32, Hq=32, Hkv=32, D=128, dtype="f16", q_dtype="f16",
            ctx_range=(512, 2048), free_frac=0.10),
    3: dict(name="Llama-3.1-70B-shaped GQA decode layer, bf16, ctx 8192",
            B=64, Hq=64, Hkv=8, D=128, dtype="bf16", q_dtype="bf16", ctx=8192),
    4: dict(name="shared-prefix copy-on-write decode, bf16",
            B=128, Hq=32, Hkv=8, D=128, dtype="bf16", q_dtype="bf16",
            prefix=384, suffix_range=(64, 1024), free_frac=0.10),
    5: dict(name="long-context fp8-E4M3 KV decode, ctx 32768",
            B=16, Hq=32, Hkv=8, D=128, dtype="fp8_e4m3", q_dtype="bf16", ctx=32768),
}


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str          # cache dtype
    q_dtype: str        # q / out / new-token dtype (new tokens use `dtype` unless fp8)
    num_blocks: int
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]
    v_scale: Optional[torch.Tensor]
    tables: List[List[int]]      # per sequence: blocks holding its cached tokens
    cached: List[int]            # tokens cached before the append
    prefix_blocks: int = 0
    seed: int = 0
    extra: dict = field(default_factory=dict)
    q_len: int = 1               # new tokens per sequence
    window: int = 0              # sliding window (0 = none)

    @property
    def new_dtype(self):
        return self.q_dtype if self.dtype == "fp8_e4m3" else self.dtype

    @property
    def context_lens(self):
        return [c + self.q_len for c in self.cached]

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.D)

    @property
    def max_blocks(self):
        return max(1, max((c + BLOCK - 1) // BLOCK for c in self.context_lens))

    def attended(self, ctx):
        """Positions some row of a sequence of length ctx attends."""
        if self.window:
            return min(ctx, self.window + self.q_len - 1)
        return ctx

    def kv_bytes(self, context_lens=None):
        """Logical bytes of K and V attention reads (+ fp8 scales): the
        positions attended (inside the window, if any), for the workload's
        context lengths or the ones given (a later step of the same
        sequences)."""
        lens = self.context_lens if context_lens is None else [int(c) for c in context_lens]
        per_tok = 2 * self.Hkv * self.D * ITEMSIZE[self.dtype]
        total = sum(self.attended(c) for c in lens) * per_tok
        if self.dtype == "fp8_e4m3":
            total += sum((c + BLOCK - 1) // BLOCK - (c - self.attended(c)) // BLOCK
                         for c in lens) * self.Hkv * 2 * 4
        return total

    def unique_kv_bytes(self):
        """Bytes of distinct blocks read (shared prefix blocks counted once)."""
        blocks = set()
        for b, c in enumerate(self.context_lens):
            nb = (c + BLOCK - 1) // BLOCK
            for j in range(min(nb, len(self.tables[b]))):
                blocks.add(self.tables[b][j])
        nb_new = sum(max(0, (c + BLOCK - 1) // BLOCK - len(self.tables[b]))
                     for b, c in enumerate(self.context_lens))
        per_block = 2 * self.Hkv * BLOCK * self.D * ITEMSIZE[self.dtype]
        return (len(blocks) + nb_new) * per_block


def _fill_normal(t_out, gen, storage, chunk=1 << 24):
    """Fills t_out (flat view) with N(0,1) rounded to `storage`."""
    flat = t_out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32)
        flat[s:e] = x.to(flat.dtype) if storage != "fp8_e4m3" else x
    return t_out


def make(spec, seed: int) -> Workload:
    """Builds a workload from a spec dict (keys as in SPECS)."""
    g = torch.Generator().manual_seed(seed)
    B, Hq, Hkv, D = spec["B"], spec["Hq"], spec["Hkv"], spec["D"]
    dtype, q_dtype = spec["dtype"], spec.get("q_dtype", spec["dtype"])
    new_dtype = q_dtype if dtype == "fp8_e4m3" else dtype

    # (1) context lengths (attended, including the appended token)
    prefix = spec.get("prefix", 0)
    if "ctx" in spec:
        ctx = spec["ctx"]
        ctx = list(ctx) if isinstance(ctx, (list, tuple)) else [ctx] * B
    elif "ctx_range" in spec:
        lo, hi = spec["ctx_range"]
        ctx = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    else:
        lo, hi = spec["suffix_range"]
        ctx = [prefix + s + 1 for s in torch.randint(lo, hi + 1, (B,), generator=g).tolist()]
    L = spec.get("q_len", 1)
    cached = [c - L for c in ctx]
    if min(cached, default=0) < 0:
        raise ValueError("context shorter than q_len")

    # (2) physical blocks
    pblocks = prefix // BLOCK
    if prefix % BLOCK:
        raise ValueError("shared prefix must be whole blocks")
    need = [(c + BLOCK - 1) // BLOCK for c in cached]
    private = [n - pblocks for n in need]
    used = pblocks + sum(private)
    if "pool" in spec:
        num_blocks = spec["pool"]
    else:
        num_blocks = used + int(math.ceil(used * spec.get("free_frac", 0.0)))
        num_blocks = max(num_blocks, used + spec.get("min_free", 0))
    if num_blocks < used:
        raise ValueError("pool too small")
    perm = torch.randperm(num_blocks, generator=g).tolist()
    shared = perm[:pblocks]
    tables, k = [], pblocks
    for b in range(B):
        tables.append(shared + perm[k:k + private[b]])
        k += private[b]

    # (3)(4) pools
    shape = (num_blocks, Hkv, BLOCK, D)
    if dtype == "fp8_e4m3":
        def fp8_pool():
            x = torch.empty(shape, dtype=torch.float32)
            _fill_normal(x, g, "fp8_e4m3")
            x = x.to(_TORCH[new_dtype]).float()            # values as new tokens carry them
            amax = x.abs().amax(dim=(2, 3))
            sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).contiguous()
            return x, (x / sc[:, :, None, None]).to(torch.float8_e4m3fn), sc
        k_vals, k_cache, k_scale = fp8_pool()
        v_vals, v_cache, v_scale = fp8_pool()
    else:
        k_cache = _fill_normal(torch.empty(shape, dtype=_TORCH[dtype]), g, dtype)
        v_cache = _fill_normal(torch.empty(shape, dtype=_TORCH[dtype]), g, dtype)
        k_vals = v_vals = None
        k_scale = v_scale = None

    # (5) queries
    qshape = (B, Hq, D) if "q_len" not in spec else (B, L, Hq, D)
    q = torch.randn(qshape, generator=g, dtype=torch.float32).to(_TORCH[q_dtype])

    # appended tokens: the pool value at positions cached .. cached + L - 1, then zeroed
    k_new = torch.empty((B, L, Hkv, D), dtype=_TORCH[new_dtype])
    v_new = torch.empty((B, L, Hkv, D), dtype=_TORCH[new_dtype])
    for b in range(B):
        for t in range(L):
            pos = cached[b] + t
            j, off = pos // BLOCK, pos % BLOCK
            if j < len(tables[b]):
                blk = tables[b][j]
            else:  # the token opens a block the block manager will pick; draw from a
                blk = perm[(used + b * L + t) % num_blocks]  # deterministic spare tile instead
            if dtype == "fp8_e4m3":
                k_new[b, t] = k_vals[blk, :, off, :].to(k_new.dtype)
                v_new[b, t] = v_vals[blk, :, off, :].to(v_new.dtype)
            else:
                k_new[b, t] = k_cache[blk, :, off, :]
                v_new[b, t] = v_cache[blk, :, off, :]
            if j < len(tables[b]):
                k_cache[blk, :, off, :] = 0
                v_cache[blk, :, off, :] = 0
    if "q_len" not in spec:
        k_new, v_new = k_new[:, 0], v_new[:, 0]
    return Workload(name=spec.get("name", "custom"), B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                    q_dtype=q_dtype, num_blocks=num_blocks, q=q, k_new=k_new, v_new=v_new,
                    k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                    tables=tables, cached=cached, prefix_blocks=pblocks, seed=seed, q_len=L,
                    window=spec.get("window", 0))


def config(index: int, **overrides) -> Workload:
    """Workload `index` (1..5) of SPECS, seed 1000 + index; keyword overrides
    (e.g. B=4) shrink it for quick checks."""
    spec = dict(SPECS[index])
    spec.update(overrides)
    return make(spec, 1000 + index)


# Prefill workloads (a prompt, or a prompt chunk after a cached prefix, per
# sequence; every new token attends causally).  "page": the pages' prefill
# benchmark shape (fp16, 16 heads, D 64, 2048 tokens, one sequence);
# "llama70b": the Llama-3.1-70B-shaped GQA layer with four 2048-token prompts;
# "chunked": four 1024-token chunks after 4096 cached positions.
PREFILL_SPECS = {
    "page": dict(n=[2048], prefix=[0], Hq=16, Hkv=16, D=64, dtype="f16"),
    "llama70b": dict(n=[2048] * 4, prefix=[0] * 4, Hq=64, Hkv=8, D=128, dtype="bf16"),
    "chunked": dict(n=[1024] * 4, prefix=[4096] * 4, Hq=64, Hkv=8, D=128, dtype="bf16"),
}


def make_prefill(seed, n, prefix, Hq, Hkv, D, dtype, free=4, stale_nan=True, window=0):
    """Paged caches holding sequences of ctx_b = prefix_b + n_b positions
    (block ids a random permutation, every value N(0,1) rounded to dtype),
    packed q [sum n, Hq, D] for the n_b new tokens with row offsets q_start,
    and NaN in every stale position past ctx_b inside a sequence's last block
    (stale_nan).  Draw order: permutation, K, V, q."""
    import numpy as np
    g = torch.Generator().manual_seed(seed)
    B = len(n)
    ctx = [p + m for p, m in zip(prefix, n)]
    need = [(c + BLOCK - 1) // BLOCK for c in ctx]
    nb = sum(need) + free
    perm = torch.randperm(nb, generator=g).tolist()
    tables, k = [], 0
    for b in range(B):
        tables.append(perm[k:k + need[b]])
        k += need[b]
    table = np.full((B, max(1, max(need))), -1, dtype=np.int32)
    for b in range(B):
        table[b, :need[b]] = tables[b]
    t = _TORCH[dtype]
    kc = _fill_normal(torch.empty((nb, Hkv, BLOCK, D), dtype=t), g, dtype)
    vc = _fill_normal(torch.empty((nb, Hkv, BLOCK, D), dtype=t), g, dtype)
    if stale_nan:
        for b in range(B):
            if ctx[b] % BLOCK:
                kc[tables[b][-1], :, ctx[b] % BLOCK:] = float("nan")
                vc[tables[b][-1], :, ctx[b] % BLOCK:] = float("nan")
    q = _fill_normal(torch.empty((sum(n), Hq, D), dtype=t), g, dtype)
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    return dict(q=q, kc=kc, vc=vc, table=table, ctx=np.array(ctx, dtype=np.int32), q_start=q_start,
                n=list(n), prefix=list(prefix), dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, window=window)


def prefill_flops(c):
    """Useful FLOPs of a prefill: 4 * D per (query head, visible position)."""
    total = 0
    for b, m in enumerate(c["n"]):
        ctx = int(c["ctx"][b])
        for i in range(m):
            lim = ctx - m + i + 1
            vis = min(lim, c["window"]) if c["window"] else lim
            total += max(0, vis)
    return 4.0 * c["D"] * c["Hq"] * total
