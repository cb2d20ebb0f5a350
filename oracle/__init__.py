"""fp64 CPU oracle for paged GQA decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never imports, links or
calls it, and it shares no code with the CUDA path: the arithmetic lives in
``pkv_oracle.c`` (plain C, IEEE double, OpenMP over (row, head)), and this
module only marshals numpy arrays into it.

Functions (each cites the page passage it follows in the C source):

- ``bf16_round(x)``          double -> bf16 bits, round-to-nearest-even, once
- ``rope_rotate(x, pos, base)`` interleaved-pair RoPE of one head vector, fp64
- ``append(...)``            new token's K (rotated) / V into its page slot
- ``gather(...)``            logically ordered K, V rows of one (row, kv head)
- ``decode(...)``            softmax(q K^T * scale) V per (row, query head)
- ``decode_partials(...)``   the same per split of ``chunk`` tokens: (o, m, l)
- ``combine(...)``           merge of binary32 partials, fp64

bf16 tensors travel as ``numpy.uint16`` bit patterns; tables as ``int32``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with gcc (-O2, no fast-math, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (
        not force
        and os.path.exists(_LIB_PATH)
        and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    ):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_long
        D = ctypes.c_double
        lib.po_bf16_to_f64.restype = D
        lib.po_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.po_f64_to_bf16_rne.restype = ctypes.c_uint16
        lib.po_f64_to_bf16_rne.argtypes = [D]
        lib.po_f64_to_bf16_array.argtypes = [P, P, L]
        lib.po_bf16_to_f64_array.argtypes = [P, P, L]
        lib.po_rope_rotate.argtypes = [P, P, I, L, D]
        lib.po_gather.restype = I
        lib.po_gather.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P]
        lib.po_append.restype = I
        lib.po_append.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, I, D, I]
        lib.po_decode.restype = I
        lib.po_decode.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, D, P]
        lib.po_decode_partials.restype = I
        lib.po_decode_partials.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, D, I, L, P, P]
        lib.po_combine.restype = I
        lib.po_combine.argtypes = [I, I, I, I, P, P, P]
        lib.po_advance.argtypes = [I, I, I, I, P, P, P, P, I, P, P, P, P]
        lib.po_prefill.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, D, P]
        lib.po_extend.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I, D, I]
        lib.po_set_threads.argtypes = [I]
        lib.po_max_threads.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def set_threads(n: int) -> None:
    _load().po_set_threads(int(n))


def max_threads() -> int:
    return int(_load().po_max_threads())


def bf16_to_f64(bits) -> np.ndarray:
    bits = _c(np.asarray(bits, dtype=np.uint16), np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().po_bf16_to_f64_array(_ptr(bits), _ptr(out), bits.size)
    return out


def bf16_round(x) -> np.ndarray:
    """Round doubles to bf16 (ties to even); returns uint16 bit patterns."""
    x = _c(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().po_f64_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def rope_rotate(x, pos: int, base: float) -> np.ndarray:
    x = _c(np.asarray(x, dtype=np.float64), np.float64)
    assert x.ndim == 1 and x.size % 2 == 0
    y = np.empty_like(x)
    _load().po_rope_rotate(_ptr(x), _ptr(y), x.size, int(pos), float(base))
    return y


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: table names a token or page outside its range")


def append(q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
           *, rope_base: float | None, rope_q: bool):
    """Return (q', k_pool', v_pool') after writing each row's new token.

    q [B,Hq,D], k_new/v_new [B,Hkv,D], pools [P,ps,Hkv,D] (uint16 bf16 bits).
    Inputs are not modified; copies are returned."""
    q = _c(q, np.uint16).copy()
    k_pool = _c(k_pool, np.uint16).copy()
    v_pool = _c(v_pool, np.uint16).copy()
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    P, ps, Hkv, D2 = k_pool.shape
    assert D2 == D and k_new.shape == (B, Hkv, D)
    rc = _load().po_append(B, Hq, Hkv, D, ps, P, _ptr(q), _ptr(k_new), _ptr(v_new),
                           _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices),
                           _ptr(kv_indptr), _ptr(seq_lens),
                           int(rope_base is not None),
                           float(rope_base or 0.0), int(bool(rope_q)))
    _check(rc, "append")
    return q, k_pool, v_pool


def extend(q, k_new, v_new, qo_indptr, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
           *, rope_base: float | None, rope_q: bool):
    """Return (q', k_pool', v_pool') after writing every row's chunk of new
    tokens (the last q_len of its seq_lens[b]) at their slots.
    q [total_q,Hq,D], k_new/v_new [total_q,Hkv,D], pools [P,ps,Hkv,D] (uint16
    bf16 bits).  Inputs are not modified; copies are returned."""
    q = _c(q, np.uint16).copy()
    k_pool = _c(k_pool, np.uint16).copy()
    v_pool = _c(v_pool, np.uint16).copy()
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    qo_indptr = _c(qo_indptr, np.int32)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    total_q, Hq, D = q.shape
    P, ps, Hkv, D2 = k_pool.shape
    B = len(seq_lens)
    assert D2 == D and k_new.shape == (total_q, Hkv, D)
    rc = _load().po_extend(B, Hq, Hkv, D, ps, P, total_q, _ptr(q), _ptr(k_new), _ptr(v_new),
                           _ptr(qo_indptr), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices),
                           _ptr(kv_indptr), _ptr(seq_lens), int(rope_base is not None),
                           float(rope_base or 0.0), int(bool(rope_q)))
    _check(rc, "extend")
    return q, k_pool, v_pool


def gather(b: int, g: int, k_pool, v_pool, kv_indices, kv_indptr, seq_lens):
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    P, ps, Hkv, D = k_pool.shape
    L = int(seq_lens[b])
    K = np.empty((L, D), dtype=np.float64)
    V = np.empty((L, D), dtype=np.float64)
    rc = _load().po_gather(b, g, Hkv, D, ps, P, _ptr(k_pool), _ptr(v_pool),
                           _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens),
                           _ptr(K), _ptr(V))
    _check(rc, "gather")
    return K, V


def decode(q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, scale: float):
    """out [B,Hq,D] float64 = softmax(q K^T * scale) V over each row's tokens."""
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_pool.shape
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().po_decode(B, Hq, Hkv, D, ps, P, _ptr(q), _ptr(k_pool), _ptr(v_pool),
                           _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens),
                           float(scale), _ptr(out))
    _check(rc, "decode")
    return out


def prefill(q, qo_indptr, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, scale: float):
    """out [total_q,Hq,D] float64: query i of row b (the last q_len of its
    seq_lens[b] tokens) attends causally up to its own position."""
    q = _c(q, np.uint16)
    qo_indptr = _c(qo_indptr, np.int32)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    total_q, Hq, D = q.shape
    B = len(seq_lens)
    P, ps, Hkv, _ = k_pool.shape
    out = np.empty((total_q, Hq, D), dtype=np.float64)
    rc = _load().po_prefill(B, Hq, Hkv, D, ps, P, total_q, _ptr(q), _ptr(qo_indptr),
                            _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices), _ptr(kv_indptr),
                            _ptr(seq_lens), float(scale), _ptr(out))
    _check(rc, "prefill")
    return out


def decode_partials(q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens, scale: float,
                    num_splits: int, chunk: int):
    """(o_part [B,Hq,S,D], ml_part [B,Hq,S,2]) float64, split s = tokens
    [s*chunk, min((s+1)*chunk, L))."""
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    kv_indices = _c(kv_indices, np.int32)
    kv_indptr = _c(kv_indptr, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_pool.shape
    o = np.empty((B, Hq, num_splits, D), dtype=np.float64)
    ml = np.empty((B, Hq, num_splits, 2), dtype=np.float64)
    rc = _load().po_decode_partials(B, Hq, Hkv, D, ps, P, _ptr(q), _ptr(k_pool),
                                    _ptr(v_pool), _ptr(kv_indices), _ptr(kv_indptr),
                                    _ptr(seq_lens), float(scale), int(num_splits),
                                    int(chunk), _ptr(o), _ptr(ml))
    _check(rc, "decode_partials")
    return o, ml


def combine(o_part, ml_part) -> np.ndarray:
    """Merge partials o_part [B,Hq,S,D], ml_part [B,Hq,S,2] -> float64 [B,Hq,D].
    binary32 inputs (what the library writes) are widened exactly."""
    o_part = np.ascontiguousarray(np.asarray(o_part), dtype=np.float64)
    ml_part = np.ascontiguousarray(np.asarray(ml_part), dtype=np.float64)
    B, Hq, S, D = o_part.shape
    assert ml_part.shape == (B, Hq, S, 2)
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().po_combine(B, Hq, D, S, _ptr(o_part), _ptr(ml_part), _ptr(out))
    _check(rc, "combine")
    return out


def advance(seq_lens, kv_indptr, kv_indices, free_pages, head: int, page_size: int,
            max_seq_len: int):
    """One decode step's metadata advance (see po_advance).  Returns
    (seq_lens, kv_indices, head, n_len, n_page, n_bad) as new int32 arrays /
    ints; the inputs are not modified."""
    sl = np.array(np.asarray(seq_lens), dtype=np.int32, copy=True)
    ind = np.array(np.asarray(kv_indices), dtype=np.int32, copy=True)
    ptr = np.ascontiguousarray(np.asarray(kv_indptr), dtype=np.int32)
    fp = np.ascontiguousarray(np.asarray(free_pages if free_pages is not None else []),
                              dtype=np.int32)
    h = np.array([head], dtype=np.int32)
    c = [ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)]
    rc = _load().po_advance(len(sl), page_size, max_seq_len, len(ind), _ptr(sl), _ptr(ptr),
                            _ptr(ind) if len(ind) else None, _ptr(fp) if len(fp) else None,
                            len(fp), _ptr(h), ctypes.byref(c[0]), ctypes.byref(c[1]),
                            ctypes.byref(c[2]))
    _check(rc, "advance")
    return sl, ind, int(h[0]), c[0].value, c[1].value, c[2].value
