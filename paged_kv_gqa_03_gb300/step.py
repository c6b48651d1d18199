"""One decode step of a paged-KV attention layer, chained through the C ABI:

  a1  host block manager: reserve each sequence's next slot (allocating a
      block or copying a shared one on write) and export tables + lengths;
  a2  paged_kv_copy_blocks for the copy-on-write pairs, if any;
  a3  paged_kv_append of the new token's K/V at its slot;
  a4-a8  paged_decode_attention (gather, scores, online softmax, p.V, merge).

Device state (caches, scales, tables, workspace) stays resident; per step
only q, k_new, v_new and the host-produced slot mapping / tables / lengths
cross to the device.  Everything is asynchronous on `stream`.
"""
import numpy as np
import torch

from . import (BlockManager, lib, paged_decode_attention, paged_decode_workspace_bytes,
               paged_kv_append, paged_kv_copy_blocks)


class DecodeStep:
    def __init__(self, k_cache, v_cache, Hq, q_dtype, max_blocks, k_scale=None, v_scale=None,
                 num_splits=0, stream=None, scale=None):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.k_scale, self.v_scale = k_scale, v_scale
        self.num_blocks, self.Hkv, _, self.D = k_cache.shape
        self.Hq, self.q_dtype, self.max_blocks = Hq, q_dtype, max_blocks
        self.num_splits = num_splits
        self.scale = 1.0 / float(np.sqrt(self.D)) if scale is None else float(scale)
        self.device = k_cache.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.bm = BlockManager(self.num_blocks)
        self.seqs = []
        self._ws = None
        self._B = None
        self._sets = []     # two pinned host buffer sets, used alternately
        self._turn = 0
        self.ncow = 0

    # -- a1 ---------------------------------------------------------------
    def adopt(self, seq, blocks, num_tokens):
        self.bm.adopt(seq, blocks, num_tokens)
        self.seqs.append(seq)

    def _buffers(self, B):
        if self._B == B:
            return
        dev, pin = self.device, torch.cuda.is_available()
        self._B = B
        self.h_seqs = np.empty(B, dtype=np.int64)
        self._sets = []
        for _ in range(2):
            self._sets.append(dict(
                slots=torch.empty(B, dtype=torch.int64, pin_memory=pin),
                pairs=torch.empty(2 * B, dtype=torch.int32, pin_memory=pin),
                table=torch.empty((B, self.max_blocks), dtype=torch.int32, pin_memory=pin),
                lens=torch.empty(B, dtype=torch.int32, pin_memory=pin),
                done=None))
        self.d_slots = torch.empty(B, dtype=torch.int64, device=dev)
        self.d_pairs = torch.empty(2 * B, dtype=torch.int32, device=dev)
        self.d_table = torch.empty((B, self.max_blocks), dtype=torch.int32, device=dev)
        self.d_lens = torch.empty(B, dtype=torch.int32, device=dev)
        n = paged_decode_workspace_bytes(B, self.Hq, self.Hkv, self.D, self.k_cache.dtype,
                                         self.q_dtype, self.num_splits)
        self._ws = torch.empty(n, dtype=torch.uint8, device=dev)

    def prepare(self, seqs=None):
        """Host part: slots, copy pairs, tables and lengths into pinned buffers.
        Returns the number of copy-on-write pairs (raises on OOM)."""
        seqs = self.seqs if seqs is None else seqs
        self._buffers(len(seqs))
        self._turn ^= 1
        hs = self._sets[self._turn]
        if hs["done"] is not None:      # the copies that last read this set have finished
            hs["done"].synchronize()
        self.h_slots, self.h_pairs, self.h_table, self.h_lens = (
            hs["slots"], hs["pairs"], hs["table"], hs["lens"])
        self.h_seqs[:] = seqs
        ncow = self.bm.append_slots_into(self.h_seqs, self.h_slots.numpy(), self.h_pairs.numpy())
        if ncow < 0:
            raise MemoryError("block manager out of blocks")
        self.ncow = ncow
        rc = lib().pkv_bm_export(self.bm._h, self.h_seqs.ctypes.data, len(seqs),
                                 self.h_table.data_ptr(), self.max_blocks, self.h_lens.data_ptr())
        if rc != 0:
            raise RuntimeError(f"export failed [{rc}]")
        return ncow

    def upload(self):
        """Host -> device copies of the step's bookkeeping (async on stream)."""
        with torch.cuda.stream(self.stream):
            self.d_slots.copy_(self.h_slots, non_blocking=True)
            self.d_table.copy_(self.h_table, non_blocking=True)
            self.d_lens.copy_(self.h_lens, non_blocking=True)
            if self.ncow:
                self.d_pairs[:2 * self.ncow].copy_(self.h_pairs[:2 * self.ncow], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.stream)
            self._sets[self._turn]["done"] = ev

    def h2d_bytes(self):
        return (self.h_slots.numel() * 8 + self.h_table.numel() * 4 + self.h_lens.numel() * 4
                + 8 * self.ncow)

    # -- a2..a8 -----------------------------------------------------------
    def launch(self, q, k_new, v_new, out):
        s = self.stream
        if self.ncow:
            paged_kv_copy_blocks(self.k_cache, self.v_cache, self.d_pairs[:2 * self.ncow].view(-1, 2),
                                 self.k_scale, self.v_scale, stream=s)
        paged_kv_append(k_new, v_new, self.k_cache, self.v_cache, self.d_slots, self.k_scale,
                        self.v_scale, stream=s)
        self.attend(q, out)

    def attend(self, q, out):
        paged_decode_attention(out, q, self.k_cache, self.v_cache, self.d_table, self.d_lens,
                               self.scale, self.k_scale, self.v_scale,
                               num_splits=self.num_splits, workspace=self._ws, stream=self.stream)

    @property
    def workspace(self):
        return self._ws

    # -- whole step as one CUDA graph ----------------------------------------
    def capture(self, h_q, h_k_new, h_v_new, h_out):
        """Captures one full step — host->device copies of q, k_new, v_new
        (pinned host tensors) and of the bookkeeping last written by
        prepare(), the append, the attention, and the device->host copy of the
        output into h_out — as a CUDA graph; replay() runs it.  Re-capture
        after prepare() when the copy pairs or buffer sets change."""
        dev = self.device
        self.g_q = torch.empty(h_q.shape, dtype=h_q.dtype, device=dev)
        self.g_k = torch.empty(h_k_new.shape, dtype=h_k_new.dtype, device=dev)
        self.g_v = torch.empty(h_v_new.shape, dtype=h_v_new.dtype, device=dev)
        self.g_out = torch.empty(h_out.shape, dtype=h_out.dtype, device=dev)
        # one eager run first: kernels are configured and tensor maps encoded
        self._graph_body(h_q, h_k_new, h_v_new, h_out)
        self.stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            self._graph_body(h_q, h_k_new, h_v_new, h_out)
        self.graph = graph
        return graph

    def _graph_body(self, h_q, h_k_new, h_v_new, h_out):
        s = self.stream
        with torch.cuda.stream(s):
            self.g_q.copy_(h_q, non_blocking=True)
            self.g_k.copy_(h_k_new, non_blocking=True)
            self.g_v.copy_(h_v_new, non_blocking=True)
            self.d_slots.copy_(self.h_slots, non_blocking=True)
            self.d_table.copy_(self.h_table, non_blocking=True)
            self.d_lens.copy_(self.h_lens, non_blocking=True)
            if self.ncow:
                self.d_pairs[:2 * self.ncow].copy_(self.h_pairs[:2 * self.ncow], non_blocking=True)
        self.launch(self.g_q, self.g_k, self.g_v, self.g_out)
        with torch.cuda.stream(s):
            h_out.copy_(self.g_out, non_blocking=True)

    def replay(self):
        with torch.cuda.stream(self.stream):
            self.graph.replay()
