"""CPU double-precision oracle for paged GQA decode attention.

TEST INFRASTRUCTURE ONLY.  This package is the reference the CUDA library is
checked against.  Only the tests, the smoke check and the benchmark's CPU
baseline may import it; the library never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (see its header for the passages each
function follows); this module only marshals numpy arrays through ctypes.
``block_table.py`` holds the pure-Python block allocator of the page
"大模型推理加速核心KV Cache 复用机制与内存布局优化" §三.

Arrays are numpy; 16-bit and 8-bit floating caches are passed as their raw
bits (uint16 / uint8 arrays) together with an explicit dtype name, so the
oracle decodes every element itself.
"""
import ctypes
import math

import numpy as np

from . import build as _build

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "fp8_e4m3": 3}
_ITEM = {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = f64
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = f64
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = f64
        L.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        L.oracle_e4m3_from_float.restype = ctypes.c_uint8
        L.oracle_kv_bytes_per_token.argtypes = [i32, i32, i32, f64]
        L.oracle_kv_bytes_per_token.restype = f64
        L.oracle_append.argtypes = [P, P, i32, P, P, P, P, i32, P, i32, i32, i32, i64, i32]
        L.oracle_append.restype = i32
        L.oracle_append_calibrated.argtypes = L.oracle_append.argtypes
        L.oracle_append_calibrated.restype = i32
        L.oracle_decode.argtypes = [P, P, P, i32, P, P, i32, P, P, P, i32, P, P,
                                    i32, i32, i32, i32, i64, i32, f64, i32]
        L.oracle_decode.restype = i32
        L.oracle_decode_multi.argtypes = [P, P, P, i32, P, P, i32, P, P, P, i32, P, P,
                                          i32, i32, i32, i32, i32, i32, i64, i32, f64, i32]
        L.oracle_decode_multi.restype = i32
        L.oracle_prefill.argtypes = [P, P, P, i32, P, P, i32, P, P, P, i32, P, P,
                                     i32, i32, i32, i32, i32, i64, i32, f64, i32]
        L.oracle_prefill.restype = i32
        L.oracle_merge.argtypes = [P, P, P, i32, i32, i32]
        L.oracle_merge.restype = None
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = i32
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _raw(a, dtype):
    """Contiguous numpy view of a tensor's raw element bits for `dtype`."""
    try:  # torch tensors (CPU) are accepted for convenience
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype in (torch.bfloat16, torch.float16):
                a = a.view(torch.int16).numpy().view(np.uint16)
            elif a.dtype == torch.float8_e4m3fn:
                a = a.view(torch.uint8).numpy()
            else:
                a = a.numpy()
    except ImportError:
        pass
    a = np.ascontiguousarray(a)
    want = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16,
            "fp8_e4m3": np.uint8}[dtype]
    if dtype == "f16" and a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError(f"expected raw {want} array for {dtype}, got {a.dtype}")
    return a


def num_threads():
    return lib().oracle_num_threads()


def f16_to_double(bits):
    L = lib()
    return np.array([L.oracle_f16_to_double(int(b)) for b in np.ravel(bits)])


def bf16_to_double(bits):
    L = lib()
    return np.array([L.oracle_bf16_to_double(int(b)) for b in np.ravel(bits)])


def e4m3_to_double(codes):
    L = lib()
    return np.array([L.oracle_e4m3_to_double(int(c)) for c in np.ravel(codes)])


def e4m3_from_float(x):
    L = lib()
    return np.array([L.oracle_e4m3_from_float(float(v)) for v in
                     np.ravel(np.asarray(x, dtype=np.float32))], dtype=np.uint8)


def kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype_bytes):
    return lib().oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim,
                                           float(dtype_bytes))


def append(k_cache, v_cache, cache_dtype, k_new, v_new, new_dtype, slot_mapping,
           k_scale=None, v_scale=None, block_size=16, inplace=False, calibrated=False):
    """Writes the new tokens into COPIES of the caches (into the given arrays
    themselves when inplace=True); returns (k_cache, v_cache, k_scale, v_scale)
    after the append.  calibrated=True: FP8 block scales follow the running
    max of the block's tokens, earlier tokens re-quantised when it grows."""
    kc = _raw(k_cache, cache_dtype)
    vc = _raw(v_cache, cache_dtype)
    if not inplace:
        kc, vc = kc.copy(), vc.copy()
    kn = _raw(k_new, new_dtype)
    vn = _raw(v_new, new_dtype)
    B, Hkv, D = kn.shape
    num_blocks = kc.shape[0]
    def _scales(x):
        if x is None:
            return None
        if inplace:
            x = _raw(x, "f32")
            return x
        return np.array(x, dtype=np.float32, copy=True)
    ks, vs = _scales(k_scale), _scales(v_scale)
    sm = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int64))
    fn = lib().oracle_append_calibrated if calibrated else lib().oracle_append
    rc = fn(_ptr(kc), _ptr(vc), DTYPES[cache_dtype], _ptr(ks), _ptr(vs),
                             _ptr(kn), _ptr(vn), DTYPES[new_dtype], _ptr(sm),
                             B, Hkv, D, num_blocks, block_size)
    if rc != 0:
        raise ValueError("oracle_append: unsupported dtype combination")
    return kc, vc, ks, vs


def decode(q, q_dtype, k_cache, v_cache, cache_dtype, block_table, context_lens,
           scale=None, k_scale=None, v_scale=None, block_size=16, t_begin=None,
           nthreads=0, with_lse=False, window=0):
    """Exact attention of each query row over its sequence's gathered cache.

    q [B, Hq, D]: one new token per sequence -> out float64 [B, Hq, D] (and
    lse [B, Hq] when with_lse).  q [B, q_len, Hq, D]: q_len new tokens per
    sequence, each seeing the positions up to its own -> out [B, q_len, Hq, D]
    (lse [B, q_len, Hq]).  window > 0: each row sees only the `window` most
    recent positions up to its own."""
    qr = _raw(q, q_dtype)
    kc = _raw(k_cache, cache_dtype)
    vc = _raw(v_cache, cache_dtype)
    multi = qr.ndim == 4
    if multi:
        B, q_len, Hq, D = qr.shape
    else:
        (B, Hq, D), q_len = qr.shape, 1
    num_blocks, Hkv = kc.shape[0], kc.shape[1]
    if kc.shape[2] != block_size or kc.shape[3] != D:
        raise ValueError("cache shape must be [num_blocks, Hkv, block_size, D]")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    tb = None if t_begin is None else np.ascontiguousarray(np.asarray(t_begin, dtype=np.int32))
    ks = None if k_scale is None else np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32))
    vs = None if v_scale is None else np.ascontiguousarray(np.asarray(v_scale, dtype=np.float32))
    if cache_dtype == "fp8_e4m3" and (ks is None or vs is None):
        raise ValueError("fp8 cache needs k_scale and v_scale")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty(qr.shape, dtype=np.float64)
    lse = np.empty(qr.shape[:-1], dtype=np.float64)
    if multi or window:
        rc = lib().oracle_decode_multi(_ptr(out), _ptr(lse), _ptr(qr), DTYPES[q_dtype], _ptr(kc),
                                       _ptr(vc), DTYPES[cache_dtype], _ptr(ks), _ptr(vs), _ptr(bt),
                                       bt.shape[1], _ptr(cl), _ptr(tb), B, q_len, int(window), Hq,
                                       Hkv, D, num_blocks, block_size, float(scale), int(nthreads))
    else:
        rc = lib().oracle_decode(_ptr(out), _ptr(lse), _ptr(qr), DTYPES[q_dtype], _ptr(kc),
                                 _ptr(vc), DTYPES[cache_dtype], _ptr(ks), _ptr(vs), _ptr(bt),
                                 bt.shape[1], _ptr(cl), _ptr(tb), B, Hq, Hkv, D, num_blocks,
                                 block_size, float(scale), int(nthreads))
    if rc == -1:
        raise ValueError("oracle_decode: Hq must be a multiple of Hkv")
    if rc == -2:
        raise ValueError("oracle_decode: block table entry out of range")
    return (out, lse) if with_lse else out


def prefill(q, q_dtype, k_cache, v_cache, cache_dtype, block_table, context_lens, q_start,
            scale=None, k_scale=None, v_scale=None, block_size=16, nthreads=0, with_lse=False,
            window=0):
    """Causal attention of each sequence's new tokens: q [total, Hq, D] holds
    sequence b's n_b = q_start[b+1] - q_start[b] new tokens from row
    q_start[b]; they are its n_b newest positions.  Returns out float64
    [total, Hq, D] (and lse [total, Hq])."""
    qr = _raw(q, q_dtype)
    kc = _raw(k_cache, cache_dtype)
    vc = _raw(v_cache, cache_dtype)
    total, Hq, D = qr.shape
    num_blocks, Hkv = kc.shape[0], kc.shape[1]
    if kc.shape[2] != block_size or kc.shape[3] != D:
        raise ValueError("cache shape must be [num_blocks, Hkv, block_size, D]")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    qs = np.ascontiguousarray(np.asarray(q_start, dtype=np.int32))
    B = len(cl)
    if len(qs) != B + 1 or qs[0] != 0 or qs[-1] != total or np.any(np.diff(qs) < 0):
        raise ValueError("q_start must be [B+1] offsets from 0 to the row count")
    ks = None if k_scale is None else np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32))
    vs = None if v_scale is None else np.ascontiguousarray(np.asarray(v_scale, dtype=np.float32))
    if cache_dtype == "fp8_e4m3" and (ks is None or vs is None):
        raise ValueError("fp8 cache needs k_scale and v_scale")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty(qr.shape, dtype=np.float64)
    lse = np.empty(qr.shape[:-1], dtype=np.float64)
    rc = lib().oracle_prefill(_ptr(out), _ptr(lse), _ptr(qr), DTYPES[q_dtype], _ptr(kc), _ptr(vc),
                              DTYPES[cache_dtype], _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1],
                              _ptr(cl), _ptr(qs), B, int(window), Hq, Hkv, D, num_blocks,
                              block_size, float(scale), int(nthreads))
    if rc == -1:
        raise ValueError("oracle_prefill: Hq must be a multiple of Hkv")
    if rc == -2:
        raise ValueError("oracle_prefill: block table entry out of range")
    return (out, lse) if with_lse else out


def merge(o_parts, lse_parts):
    """o_parts [R, S, D], lse_parts [R, S] (float64) -> out [R, D]."""
    o = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    R, S, D = o.shape
    out = np.empty((R, D), dtype=np.float64)
    lib().oracle_merge(_ptr(out), _ptr(o), _ptr(l), R, S, D)
    return out
