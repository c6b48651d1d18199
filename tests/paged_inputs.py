"""Test-side construction of small paged caches from contiguous per-sequence
K/V, so that an oracle result over the paged layout can be compared with a
library attention over the contiguous source it was scattered from."""
import numpy as np
import torch


def scatter(kv_list, Hkv, D, block_size, num_blocks, perm, dtype=torch.float64):
    """kv_list: per sequence a [T_b, Hkv, D] tensor.  Places sequence b's token
    t in block perm-chosen for (b, t // block_size).  Returns (pool
    [num_blocks, Hkv, block_size, D], tables list, max_blocks)."""
    pool = torch.randn((num_blocks, Hkv, block_size, D), dtype=torch.float64,
                       generator=torch.Generator().manual_seed(99)).to(dtype)
    tables, k = [], 0
    for x in kv_list:
        T = x.shape[0]
        nb = (T + block_size - 1) // block_size
        tbl = [int(perm[k + j]) for j in range(nb)]
        k += nb
        for t in range(T):
            pool[tbl[t // block_size], :, t % block_size, :] = x[t].to(dtype)
        tables.append(tbl)
    max_blocks = max(1, max(len(t) for t in tables))
    return pool, tables, max_blocks


def dense_table(tables, max_blocks, fill=-1):
    bt = np.full((len(tables), max_blocks), fill, dtype=np.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = t
    return bt


def sdpa_reference(q, ks, vs, scale):
    """q [B, Hq, D] float64; ks/vs per sequence [T_b, Hkv, D] float64.
    Returns [B, Hq, D] from torch's scaled_dot_product_attention."""
    B, Hq, D = q.shape
    out = torch.empty((B, Hq, D), dtype=torch.float64)
    for b in range(B):
        K, V = ks[b], vs[b]
        Hkv = K.shape[1]
        G = Hq // Hkv
        Kx = K.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, T, D]
        Vx = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b][:, None, :], Kx, Vx, scale=scale)
        out[b] = o[:, 0, :]
    return out
