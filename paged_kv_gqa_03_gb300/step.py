"""One decode step of a paged-KV attention layer, chained through the C ABI:

  a1  host block manager: reserve each sequence's next slot (allocating a
      block or copying a shared one on write) and export tables + lengths;
  a2  paged_kv_copy_blocks for the copy-on-write pairs, if any;
  a3  paged_kv_append of the new token's K/V at its slot;
  a4-a8  paged_decode_attention (gather, scores, online softmax, p.V, merge).

With q_len > 1 every sequence appends q_len tokens per step (slots in order)
and attends them causally (the verify step of speculative decoding): q, out
are [B, q_len, Hq, D] and k_new, v_new [B, q_len, Hkv, D].  With a sliding
window W each row attends its W most recent positions, and a1 first releases
the blocks that no token of the step (or later) can see, so a sequence holds
at most ceil((W + q_len - 1) / 16) + 1 blocks.

Device state (caches, scales, workspace) stays resident.  Per step only q,
k_new, v_new and the host-produced slot mapping / copy pairs / tables /
lengths cross to the device, all from ONE pinned staging buffer with one copy
(two staging buffers alternate so the host can prepare step n+1 while step n's
copy is in flight).  Everything is asynchronous on `stream`.
"""
import numpy as np
import torch

from . import (BlockManager, lib, paged_decode_attention, paged_decode_workspace_bytes,
               paged_kv_append, paged_kv_copy_blocks, pkv_copy)

_ALIGN = 256


class _Staging:
    """One contiguous byte buffer with typed sections at 256-byte offsets."""

    def __init__(self, layout, total, device, pin):
        if device.type == "cuda":
            self.buf = torch.empty(total, dtype=torch.uint8, device=device)
        else:
            self.buf = torch.empty(total, dtype=torch.uint8, pin_memory=pin)
        self.views = {}
        for name, (off, shape, dtype) in layout.items():
            n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
            self.views[name] = self.buf[off:off + n].view(dtype).view(shape)
        self.done = None   # event recorded after the last copy out of this buffer
        self.replayed = None  # the event run() records after each graph replay

    def __getitem__(self, name):
        return self.views[name]


class DecodeStep:
    def __init__(self, k_cache, v_cache, Hq, q_dtype, max_blocks, k_scale=None, v_scale=None,
                 num_splits=0, stream=None, scale=None, q_len=1, window=0, calibrated=False):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.k_scale, self.v_scale = k_scale, v_scale
        self.num_blocks, self.Hkv, _, self.D = k_cache.shape
        self.Hq, self.q_dtype, self.max_blocks = Hq, q_dtype, max_blocks
        self.new_dtype = q_dtype if k_cache.dtype == torch.float8_e4m3fn else k_cache.dtype
        self.num_splits = num_splits
        self.q_len = q_len
        self.window = window
        self.calibrated = calibrated
        self.scale = 1.0 / float(np.sqrt(self.D)) if scale is None else float(scale)
        self.device = k_cache.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.bm = BlockManager(self.num_blocks)
        self.seqs = []
        self._ws = None
        self._B = None
        self._turn = 0
        self.ncow = 0
        self.graph = None
        self._calls = {}    # marshalled C calls (Prepared), keyed by their buffers
        self._graphs = {}   # run(): one captured step per (staging buffer, output)
        self._ran = False

    # -- buffers ---------------------------------------------------------------
    def _layout(self, B):
        L = self.q_len
        rows = (B, self.Hq, self.D) if L == 1 else (B, L, self.Hq, self.D)
        kv = (B, self.Hkv, self.D) if L == 1 else (B, L, self.Hkv, self.D)
        sections = [("q", rows, self.q_dtype),
                    ("k_new", kv, self.new_dtype),
                    ("v_new", kv, self.new_dtype),
                    ("slots", (B * L,), torch.int64),
                    ("pairs", (2 * B * L,), torch.int32),
                    ("table", (B, self.max_blocks), torch.int32),
                    ("lens", (B,), torch.int32)]
        layout, off = {}, 0
        for name, shape, dtype in sections:
            layout[name] = (off, shape, dtype)
            n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
            off = (off + n + _ALIGN - 1) // _ALIGN * _ALIGN
        self._io_bytes = layout["slots"][0]           # q, k_new, v_new
        self._book_bytes = off - layout["slots"][0]   # slots .. lens
        return layout, off

    def _buffers(self, B):
        if self._B == B:
            return
        self._B = B
        self._calls.clear()     # their buffers are about to be replaced
        self._graphs.clear()
        layout, total = self._layout(B)
        pin = torch.cuda.is_available()
        self._host = [_Staging(layout, total, torch.device("cpu"), pin) for _ in range(2)]
        self._dev = _Staging(layout, total, self.device, False)
        self.h_seqs = np.empty(B, dtype=np.int64)
        self.h_tok_seqs = np.empty(B * self.q_len, dtype=np.int64)
        self.d_q, self.d_k_new, self.d_v_new = self._dev["q"], self._dev["k_new"], self._dev["v_new"]
        self.d_slots, self.d_pairs = self._dev["slots"], self._dev["pairs"]
        self.d_table, self.d_lens = self._dev["table"], self._dev["lens"]
        self._select(self._turn)
        n = paged_decode_workspace_bytes(B, self.Hq, self.Hkv, self.D, self.k_cache.dtype,
                                         self.q_dtype, self.num_splits, q_len=self.q_len)
        self._ws = torch.empty(n, dtype=torch.uint8, device=self.device)

    def _select(self, turn):
        hs = self._host[turn]
        self.h_q, self.h_k_new, self.h_v_new = hs["q"], hs["k_new"], hs["v_new"]
        self.h_slots, self.h_pairs = hs["slots"], hs["pairs"]
        self.h_table, self.h_lens = hs["table"], hs["lens"]

    # -- a1 ----------------------------------------------------------------------
    def adopt(self, seq, blocks, num_tokens):
        self.bm.adopt(seq, blocks, num_tokens)
        self.seqs.append(seq)

    def prepare(self, seqs=None):
        """Host part of a step: switches to the other staging buffer (waiting
        for the copy that last read it), then writes the slots, copy pairs,
        tables and lengths of q_len new tokens per sequence into it.  Returns
        the number of copy-on-write pairs (raises on OOM)."""
        seqs = self.seqs if seqs is None else seqs
        self._buffers(len(seqs))
        self._turn ^= 1
        if self._host[self._turn].done is not None:
            self._host[self._turn].done.synchronize()
        self._select(self._turn)
        self.h_seqs[:] = seqs
        if self.window:
            for seq in seqs:
                self.bm.release_outside_window(int(seq), self.window)
        if self.q_len == 1:
            tok_seqs = self.h_seqs
        else:
            tok_seqs = self.h_tok_seqs
            tok_seqs.reshape(-1, self.q_len)[:] = self.h_seqs[:, None]
        ncow = self.bm.append_slots_into(tok_seqs, self.h_slots.numpy(), self.h_pairs.numpy())
        if ncow < 0:
            raise MemoryError("block manager out of blocks")
        self.ncow = ncow
        rc = lib().pkv_bm_export(self.bm._h, self.h_seqs.ctypes.data, len(seqs),
                                 self.h_table.data_ptr(), self.max_blocks, self.h_lens.data_ptr())
        if rc != 0:
            raise RuntimeError(f"export failed [{rc}]")
        return ncow

    def _copy_in(self, with_inputs):
        """One host->device copy of the current staging buffer (the step's
        bookkeeping, and q / k_new / v_new when with_inputs)."""
        hs = self._host[self._turn]
        lo = 0 if with_inputs else self._io_bytes
        hi = self._io_bytes + self._book_bytes
        pkv_copy(self._dev.buf[lo:hi], hs.buf[lo:hi], stream=self.stream)
        with torch.cuda.stream(self.stream):
            if not torch.cuda.is_current_stream_capturing():
                ev = torch.cuda.Event()
                ev.record(self.stream)
                hs.done = ev

    def upload(self):
        """Copies the bookkeeping written by prepare() to the device."""
        self._copy_in(with_inputs=False)

    def h2d_bytes(self, with_inputs=True):
        return (self._io_bytes if with_inputs else 0) + self._book_bytes

    # -- a2..a8 ------------------------------------------------------------------
    def launch(self, q, k_new, v_new, out):
        """Runs a2..a8 with device tensors q, k_new, v_new (bookkeeping from
        the last upload())."""
        s = self.stream
        if self.ncow:
            paged_kv_copy_blocks(self.k_cache, self.v_cache, self.d_pairs[:2 * self.ncow].view(-1, 2),
                                 self.k_scale, self.v_scale, stream=s)
        key = ("append", k_new.data_ptr(), v_new.data_ptr(), self.d_slots.data_ptr())
        call = self._calls.get(key)
        if call is None:
            if self.q_len > 1:
                k_new = k_new.view(-1, self.Hkv, self.D)
                v_new = v_new.view(-1, self.Hkv, self.D)
            call = self._remember(key, paged_kv_append(
                k_new, v_new, self.k_cache, self.v_cache, self.d_slots, self.k_scale, self.v_scale,
                stream=s, calibrated=self.calibrated, prepare=True))
        call()
        self.attend(q, out)

    def attend(self, q, out):
        """a4-a8 on the current bookkeeping.  The C call's arguments are
        marshalled once per (q, out) pair and reused."""
        key = ("attend", q.data_ptr(), out.data_ptr(), self.d_table.data_ptr())
        call = self._calls.get(key)
        if call is None:
            call = self._remember(key, paged_decode_attention(
                out, q, self.k_cache, self.v_cache, self.d_table, self.d_lens, self.scale,
                self.k_scale, self.v_scale, num_splits=self.num_splits, workspace=self._ws,
                stream=self.stream, window=self.window, prepare=True))
        call()

    def _remember(self, key, call):
        if len(self._calls) >= 8:
            self._calls.clear()
        self._calls[key] = call
        return call

    @property
    def workspace(self):
        return self._ws

    # -- a whole step from host memory as one CUDA graph ---------------------------
    def capture(self, h_out):
        """Captures one full step from the current staging buffer — one
        host->device copy of q, k_new, v_new (written into h_q / h_k_new /
        h_v_new) and the bookkeeping, the append, and the attention writing
        its output straight into the pinned tensor h_out over the host link
        (no separate device->host copy) — as a CUDA graph; replay() runs it.
        Re-capture after a prepare() that switches staging buffers or changes
        the copy pairs."""
        if not h_out.is_pinned():
            raise ValueError("h_out must be pinned host memory")
        self.g_out = h_out
        self._graph_body(h_out)          # eager once: kernels configured, tensor maps encoded
        self.stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            self._graph_body(h_out)
        self.graph = graph
        return graph

    def _graph_body(self, h_out):
        self._copy_in(with_inputs=True)
        self.launch(self.d_q, self.d_k_new, self.d_v_new, h_out)

    # -- a serving loop from host memory ----------------------------------------
    def stage_inputs(self, q, k_new, v_new, both=False):
        """Writes a step's q, k_new, v_new (host tensors) into the current
        staging buffer (both=True: into both buffers)."""
        for t in ((0, 1) if both else (self._turn,)):
            hs = self._host[t]
            hs["q"].copy_(q)
            hs["k_new"].copy_(k_new)
            hs["v_new"].copy_(v_new)

    def run(self, h_out):
        """Issues one whole step from host memory, asynchronously: the copy of
        the current staging buffer (inputs and the bookkeeping of the last
        prepare()), the append and the attention writing into the pinned
        tensor h_out.  Each staging buffer has a CUDA graph of its own,
        captured on first use, so a loop can run step n from one buffer
        while prepare() writes step n + 1 into the other:

            step.prepare(); step.run(h_out)
            while serving:
                step.prepare()            # a1 of the next step, on the host
                stream.synchronize()      # this step's output is in h_out
                ...read h_out, stage the next inputs...
                step.run(h_out)

        The first step runs eagerly (it configures the kernels and encodes
        their tensor maps outside any capture), and so does a step with
        copy-on-write pairs (rare): the graphs hold no block copy.

        A loop may also keep one step queued ahead of the host (two pinned
        output tensors alternating): issue step n, wait for step n - 1 and
        read its output, then prepare() step n + 1 — prepare() waits for the
        step that last read the staging buffer it switches to."""
        if not h_out.is_pinned():
            raise ValueError("h_out must be pinned host memory")
        if self.stream.cuda_stream == 0:
            raise ValueError("run() captures CUDA graphs: give the DecodeStep a non-default stream")
        if self.ncow or not self._ran:
            self._graph_body(h_out)
            self._ran = True
            return
        key = (self._turn, h_out.data_ptr())
        graph = self._graphs.get(key)
        if graph is None:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=self.stream):
                self._graph_body(h_out)
            self._graphs[key] = graph
        with torch.cuda.stream(self.stream):
            graph.replay()
        # the graph's copy out of this staging buffer is done once the step
        # is: prepare() waits for it before rewriting the buffer
        hs = self._host[self._turn]
        if hs.replayed is None:
            hs.replayed = torch.cuda.Event()
        hs.replayed.record(self.stream)
        hs.done = hs.replayed

    def replay(self):
        with torch.cuda.stream(self.stream):
            self.graph.replay()
