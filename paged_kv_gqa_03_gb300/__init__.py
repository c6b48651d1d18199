"""Python binding of libpagedkv.so — paged GQA decode attention for sm_103a.

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels (or, for the block manager, its native host code).
PyTorch supplies device memory and streams.  Importing this package fails with
ImportError when the library has not been built — there is no fallback.

The function names are those of the C ABI in include/pagedkv.h, whose comments
define each operation, its layouts and its errors.
"""
import ctypes
import os

__all__ = [
    "PagedKVError", "paged_kv_append", "paged_decode_workspace_bytes",
    "paged_decode_attention", "paged_prefill_attention", "paged_decode_status", "paged_decode_merge",
    "paged_decode_attention_static", "paged_decode_static_status",
    "paged_kv_copy_blocks", "pkv_copy", "pkv_status_string", "pkv_version", "pkv_set_route",
    "pkv_get_route", "pkv_test_stall_next", "BlockManager", "Prepared",
    "DTYPE_CODES", "LIB_PATH", "lib",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libpagedkv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python paged_kv_gqa_03_gb300/build.py, or __graft_entry__.build())")

_P, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_L = ctypes.CDLL(LIB_PATH)


def _sig(name, res, *args):
    fn = getattr(_L, name)
    fn.restype = res
    fn.argtypes = list(args)
    return fn


_sig("paged_kv_append", _i32, _P, _P, _i32, _P, _P, _i32, _P, _P, _P, _i32, _i32, _i32, _i64, _P)
_sig("paged_kv_append_calibrated", _i32, _P, _P, _i32, _P, _P, _i32, _P, _P, _P, _i32, _i32, _i32, _i64, _P)
_sig("paged_decode_workspace_bytes", _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
     ctypes.POINTER(_sz))
_sig("paged_decode_attention", _i32, _P, _P, _i32, _P, _P, _i32, _P, _P, _P, _i32, _P,
     _i32, _i32, _i32, _i32, _i64, ctypes.c_float, _i32, _P, _sz, _P)
_sig("paged_decode_multi_workspace_bytes", _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
     ctypes.POINTER(_sz))
_sig("paged_decode_attention_multi", _i32, _P, _P, _i32, _P, _P, _i32, _P, _P, _P, _i32, _P,
     _i32, _i32, _i32, _i32, _i32, _i32, _i64, ctypes.c_float, _i32, _P, _sz, _P)
_sig("paged_prefill_attention", _i32, _P, _P, _i32, _P, _P, _i32, _P, _i32, _P, _P,
     _i32, _i32, _i32, _i32, _i32, _i64, ctypes.c_float, _i32, _P, _P)
_sig("paged_decode_status", _i32, _P, _sz, _P, ctypes.POINTER(_i32))
_sig("paged_decode_attention_static", _i32, _P, _P, _i32, _P, _P, _i32, _P, _P, _P, _i32, _P,
     _i32, _i32, _i32, _i32, _i64, ctypes.c_float, _i32, _P)
_sig("paged_decode_static_status", _i32, _P, ctypes.POINTER(_i32))
_sig("paged_decode_merge", _i32, _P, _i32, _P, _P, _i32, _i32, _i32, _i32, _P)
_sig("paged_kv_copy_blocks", _i32, _P, _P, _i32, _P, _P, _P, _i32, _i32, _i32, _i64, _P)
_sig("pkv_copy", _i32, _P, _P, _sz, _P)
_sig("pkv_status_string", ctypes.c_char_p, _i32)
_sig("pkv_last_cuda_error", _i32)
_sig("pkv_version", _i32)
_sig("pkv_set_route", _i32, _i32, _i32)
_sig("pkv_get_route", _i32, _i32)
_sig("pkv_test_stall_next", _i32, _i32, ctypes.c_uint64)
_sig("pkv_bm_create", _P, _i64)
_sig("pkv_bm_destroy", None, _P)
_sig("pkv_bm_allocate", _i32, _P, _i64, _i64)
_sig("pkv_bm_adopt", _i32, _P, _i64, _P, _i32, _i64)
_sig("pkv_bm_fork", _i32, _P, _i64, _i64)
_sig("pkv_bm_free", _i32, _P, _i64)
_sig("pkv_bm_release_window", _i32, _P, _i64, _i64, ctypes.POINTER(_i64))
_sig("pkv_bm_append_slots", _i32, _P, _P, _i32, _P, _P, ctypes.POINTER(_i32))
_sig("pkv_bm_export", _i32, _P, _P, _i32, _P, _i32, _P)
_sig("pkv_bm_num_free", _i64, _P)
_sig("pkv_bm_refcount", _i32, _P, _i64)
_sig("pkv_bm_num_tokens", _i64, _P, _i64)

PKV_OK, PKV_EINVAL, PKV_EUNSUPPORTED, PKV_EWORKSPACE = 0, -1, -2, -3
PKV_ECUDA, PKV_ETIMEOUT, PKV_EOOM, PKV_ERANGE, PKV_ENOTFOUND = -4, -5, -6, -7, -8
PKV_FLAG_TIMEOUT, PKV_FLAG_BAD_LEN, PKV_FLAG_BAD_BLOCK, PKV_FLAG_RANGE = 1, 2, 4, 8
PKV_STATIC_SCRATCH_BYTES = 16 << 20


def lib():
    """The loaded ctypes library (raw C ABI)."""
    return _L


class PagedKVError(RuntimeError):
    def __init__(self, status, where):
        msg = _L.pkv_status_string(status).decode()
        if status == PKV_ECUDA:
            msg += f" (cudaError {_L.pkv_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")
        self.status = status


def _check(status, where):
    if status != PKV_OK:
        raise PagedKVError(status, where)


def pkv_status_string(status):
    return _L.pkv_status_string(status).decode()


def pkv_version():
    return _L.pkv_version()


# Kernel-route decisions that pkv_set_route can force (include/pagedkv.h).
ROUTES = {"multi_query": (0, ("auto", "transposed", "prefill", "units")),
          "prefill": (1, ("auto", "persistent", "tiles"))}


def pkv_set_route(which, choice):
    """Forces one kernel-route decision process-wide ("multi_query":
    auto / transposed / prefill / units; "prefill": auto / persistent /
    tiles); returns the previous choice.  "auto" restores the library's rule."""
    idx, names = ROUTES[which]
    prev = names[_L.pkv_get_route(idx)]
    _check(_L.pkv_set_route(idx, names.index(choice)), "pkv_set_route")
    return prev


def pkv_test_stall_next(which, limit_ns):
    """Failure-path test hook: the next call that launches the "decode" or
    "prefill" kernel family runs out a wait on a barrier nothing completes
    (every wait of that call limited to limit_ns) and reports
    PKV_FLAG_TIMEOUT; see include/pagedkv.h."""
    _check(_L.pkv_test_stall_next({"decode": 0, "prefill": 1}[which], int(limit_ns)),
           "pkv_test_stall_next")


def pkv_get_route(which):
    idx, names = ROUTES[which]
    return names[_L.pkv_get_route(idx)]


def _torch():
    import torch
    return torch


def _dtype_codes():
    torch = _torch()
    return {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.float8_e4m3fn: 3}


DTYPE_CODES = None


def _code(t):
    global DTYPE_CODES
    if DTYPE_CODES is None:
        DTYPE_CODES = _dtype_codes()
    try:
        return DTYPE_CODES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _out(t):
    """The output pointer of a decode call: a CUDA tensor, or pinned host
    memory that the kernels write directly (see include/pagedkv.h)."""
    if t.is_cuda:
        return _dev(t, "out")
    if not t.is_pinned():
        raise ValueError("out must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError("out must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Prepared:
    """One C call with its arguments marshalled once (returned by the calls
    below when given prepare=True): calling it issues the call again on the
    same buffers and stream, for a decode loop that runs the same step every
    iteration.  The buffers must stay alive and keep their addresses."""

    __slots__ = ("fn", "args", "name")

    def __init__(self, fn, args, name):
        self.fn, self.args, self.name = fn, args, name

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != PKV_OK:
            raise PagedKVError(rc, self.name)


def paged_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None,
                    stream=None, calibrated=False, prepare=False):
    """Writes k_new/v_new [B, Hkv, D] into the caches [num_blocks, Hkv, 16, D]
    at slot_mapping[b] (int64; < 0 skips).  calibrated=True: FP8 block scales
    follow the block's running max (paged_kv_append_calibrated)."""
    torch = _torch()
    B, Hkv, D = k_new.shape
    fn = _L.paged_kv_append_calibrated if calibrated else _L.paged_kv_append
    args = (_dev(k_new, "k_new"), _dev(v_new, "v_new"), _code(k_new),
            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _code(k_cache),
            _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
            _dev(slot_mapping, "slot_mapping", torch.int64), B, Hkv, D, k_cache.shape[0],
            _stream(stream))
    if prepare:
        return Prepared(fn, args, "paged_kv_append")
    _check(fn(*args), "paged_kv_append")


def paged_decode_workspace_bytes(B, Hq, Hkv, D, cache_dtype, q_dtype, num_splits=0, q_len=1):
    """Workspace size for paged_decode_attention (q_len new tokens per
    sequence) on the current device.  dtypes are torch dtypes or C codes."""
    conv = lambda d: d if isinstance(d, int) else _code(_torch().empty(0, dtype=d))
    out = _sz(0)
    if q_len == 1:
        rc = _L.paged_decode_workspace_bytes(B, Hq, Hkv, D, conv(cache_dtype), conv(q_dtype),
                                             num_splits, ctypes.byref(out))
    else:
        rc = _L.paged_decode_multi_workspace_bytes(B, q_len, Hq, Hkv, D, conv(cache_dtype),
                                                   conv(q_dtype), num_splits, ctypes.byref(out))
    _check(rc, "paged_decode_workspace_bytes")
    return out.value


def paged_decode_attention(out, q, k_cache, v_cache, block_table, context_lens, scale,
                           k_scale=None, v_scale=None, num_splits=0, workspace=None, stream=None,
                           window=0, prepare=False):
    """out[b, hq] = softmax(scale * q[b, hq] . K_b^T) V_b over the paged cache.

    q, out [B, Hq, D]: one new token per sequence (paged_decode_attention).
    q, out [B, q_len, Hq, D]: q_len new tokens per sequence, token i seeing
    the cache up to its own position (paged_decode_attention_multi).
    window > 0: each row sees only its `window` most recent positions.
    workspace: a uint8 CUDA tensor of paged_decode_workspace_bytes(...) bytes;
    allocated here (by torch) when None.  prepare=True returns the call as a
    Prepared object instead of issuing it."""
    torch = _torch()
    if q.dim() == 4:
        B, q_len, Hq, D = q.shape
    else:
        (B, Hq, D), q_len = q.shape, 1
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out shape {tuple(out.shape)} != q shape {tuple(q.shape)}")
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    if workspace is None:
        n = paged_decode_workspace_bytes(B, Hq, Hkv, D, _code(k_cache), _code(q), num_splits,
                                         q_len=q_len)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    args = (_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _code(k_cache), _dev(k_scale, "k_scale", torch.float32),
            _dev(v_scale, "v_scale", torch.float32), _dev(block_table, "block_table", torch.int32),
            block_table.shape[1], _dev(context_lens, "context_lens", torch.int32))
    tail = (num_blocks, float(scale), num_splits, _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream))
    if q.dim() == 4 or window:
        fn, name = _L.paged_decode_attention_multi, "paged_decode_attention_multi"
        full = (_out(out), _dev(q, "q"), _code(q), *args, B, q_len, int(window), Hq, Hkv, D, *tail)
    else:
        fn, name = _L.paged_decode_attention, "paged_decode_attention"
        full = (_out(out), _dev(q, "q"), _code(q), *args, B, Hq, Hkv, D, *tail)
    if prepare:
        return Prepared(fn, full, name)
    _check(fn(*full), name)
    return workspace


def paged_prefill_attention(out, q, k_cache, v_cache, block_table, context_lens, q_start, max_q_len,
                            scale, window=0, status=None, stream=None):
    """Causal attention of each sequence's new tokens over its paged cache
    (tensor cores).  q, out [total, Hq, D]; q_start int32 [B+1] row offsets;
    max_q_len >= every sequence's new-token count; status: optional int32
    CUDA tensor that receives the PKV_FLAG_* bits."""
    torch = _torch()
    total, Hq, D = q.shape
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out shape {tuple(out.shape)} != q shape {tuple(q.shape)}")
    B = q_start.shape[0] - 1
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    _check(_L.paged_prefill_attention(
        _out(out), _dev(q, "q"), _code(q), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _code(k_cache), _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev(context_lens, "context_lens", torch.int32), _dev(q_start, "q_start", torch.int32),
        B, int(max_q_len), Hq, Hkv, D, num_blocks, float(scale), int(window),
        _dev(status, "status", torch.int32), _stream(stream)), "paged_prefill_attention")


def paged_decode_status(workspace, stream=None):
    """Synchronises the stream; returns the PKV_FLAG_* bits the last decode
    recorded in `workspace` (raises on a timeout or range flag)."""
    flags = _i32(0)
    rc = _L.paged_decode_status(_dev(workspace, "workspace"),
                                workspace.numel() * workspace.element_size(), _stream(stream),
                                ctypes.byref(flags))
    if rc not in (PKV_OK, PKV_ETIMEOUT, PKV_ERANGE):
        _check(rc, "paged_decode_status")
    return rc, flags.value


def paged_decode_attention_static(out, q, k_cache, v_cache, block_table, context_lens, scale,
                                  k_scale=None, v_scale=None, num_splits=0, stream=None):
    """paged_decode_attention (one new token per sequence, q, out [B, Hq, D])
    on the scratch array the library keeps on each GPU instead of a caller's
    workspace, for callers that cannot allocate device memory.  Calls on one
    GPU share that array: they must not overlap on the GPU."""
    torch = _torch()
    B, Hq, D = q.shape
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out shape {tuple(out.shape)} != q shape {tuple(q.shape)}")
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    _check(_L.paged_decode_attention_static(
        _out(out), _dev(q, "q"), _code(q), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _code(k_cache), _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev(context_lens, "context_lens", torch.int32), B, Hq, Hkv, D, num_blocks, float(scale),
        num_splits, _stream(stream)), "paged_decode_attention_static")


def paged_decode_static_status(stream=None):
    """paged_decode_status for the static scratch of the current device:
    (status, PKV_FLAG_* bits) of the last paged_decode_attention_static."""
    flags = _i32(0)
    rc = _L.paged_decode_static_status(_stream(stream), ctypes.byref(flags))
    if rc not in (PKV_OK, PKV_ETIMEOUT, PKV_ERANGE):
        _check(rc, "paged_decode_static_status")
    return rc, flags.value


def paged_decode_merge(out, o_partial, lse, stream=None):
    """out [B, Hq, D] from o_partial [B, Hq, S, D] fp32 and lse [B, Hq, S] fp32."""
    torch = _torch()
    B, Hq, S, D = o_partial.shape
    _check(_L.paged_decode_merge(_dev(out, "out"), _code(out),
                                 _dev(o_partial, "o_partial", torch.float32),
                                 _dev(lse, "lse", torch.float32), B, Hq, D, S, _stream(stream)),
           "paged_decode_merge")


def pkv_copy(dst, src, nbytes=None, stream=None):
    """SM-driven copy of nbytes (default: all of src) between CUDA tensors
    and/or pinned host tensors (see include/pagedkv.h)."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    n = src.numel() * src.element_size() if nbytes is None else nbytes
    _check(_L.pkv_copy(dst.data_ptr(), src.data_ptr(), n, _stream(stream)), "pkv_copy")


def paged_kv_copy_blocks(k_cache, v_cache, src_dst_pairs, k_scale=None, v_scale=None, stream=None):
    """cache[dst] = cache[src] for each (src, dst) row of the int32 [n, 2] tensor."""
    torch = _torch()
    n = src_dst_pairs.shape[0]
    _check(_L.paged_kv_copy_blocks(
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _code(k_cache),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(src_dst_pairs, "src_dst_pairs", torch.int32), n, k_cache.shape[1],
        k_cache.shape[3], k_cache.shape[0], _stream(stream)), "paged_kv_copy_blocks")


class BlockManager:
    """Host physical-block allocator (native, in libpagedkv.so): allocate /
    adopt / fork / free and per-token slot mapping with copy-on-write."""

    def __init__(self, num_blocks):
        self._h = _L.pkv_bm_create(num_blocks)
        if not self._h:
            raise MemoryError("pkv_bm_create failed")
        self.num_blocks = num_blocks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _L.pkv_bm_destroy(h)
            self._h = None

    def allocate(self, seq, num_tokens):
        rc = _L.pkv_bm_allocate(self._h, seq, num_tokens)
        if rc == PKV_EOOM:
            return False
        _check(rc, "allocate")
        return True

    def adopt(self, seq, blocks, num_tokens):
        arr = (ctypes.c_int32 * len(blocks))(*blocks)
        _check(_L.pkv_bm_adopt(self._h, seq, arr, len(blocks), num_tokens), "adopt")

    def fork(self, parent, child):
        rc = _L.pkv_bm_fork(self._h, parent, child)
        if rc == PKV_ENOTFOUND:
            return False
        _check(rc, "fork")
        return True

    def free(self, seq):
        _check(_L.pkv_bm_free(self._h, seq), "free")

    def release_outside_window(self, seq, window):
        """Releases the blocks of seq that no later token sees with this
        sliding window; returns how many table entries were released."""
        n = _i64(0)
        _check(_L.pkv_bm_release_window(self._h, seq, window, ctypes.byref(n)),
               "release_outside_window")
        return n.value

    def append_slots(self, seqs):
        """One new token per sequence: (slots list, [(src, dst), ...]) or None on OOM."""
        n = len(seqs)
        s = (ctypes.c_int64 * max(n, 1))(*seqs)
        slots = (ctypes.c_int64 * max(n, 1))()
        pairs = (ctypes.c_int32 * max(2 * n, 2))()
        ncow = _i32(0)
        rc = _L.pkv_bm_append_slots(self._h, s, n, slots, pairs, ctypes.byref(ncow))
        if rc == PKV_EOOM:
            return None
        _check(rc, "append_slots")
        return list(slots[:n]), [(pairs[2 * i], pairs[2 * i + 1]) for i in range(ncow.value)]

    def append_slots_into(self, seqs_arr, slots_arr, pairs_arr):
        """Buffer form for hot loops: numpy int64 seqs / int64 slots / int32
        [2n] pairs (host, contiguous); returns the number of copy pairs or -1 on OOM."""
        ncow = _i32(0)
        rc = _L.pkv_bm_append_slots(self._h, seqs_arr.ctypes.data, len(seqs_arr),
                                    slots_arr.ctypes.data, pairs_arr.ctypes.data, ctypes.byref(ncow))
        if rc == PKV_EOOM:
            return -1
        _check(rc, "append_slots")
        return ncow.value

    def export(self, seqs, max_blocks):
        """(table int32 [n, max_blocks] with -1 padding, context_lens int32 [n]) as numpy."""
        import numpy as np
        n = len(seqs)
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        table = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty((n,), dtype=np.int32)
        _check(_L.pkv_bm_export(self._h, s.ctypes.data, n, table.ctypes.data, max_blocks,
                                lens.ctypes.data), "export")
        return table, lens

    def num_free(self):
        return _L.pkv_bm_num_free(self._h)

    def refcount(self, block):
        return _L.pkv_bm_refcount(self._h, block)

    def num_tokens(self, seq):
        return _L.pkv_bm_num_tokens(self._h, seq)
