"""ctypes binding of libpkv (include/pkv.h) -- argument marshalling only.

Each function takes torch tensors (or raw integer device addresses), passes
their pointers and the current CUDA stream to the C entry point of the same
name, and raises :class:`PkvError` on a non-OK status.  No computation happens
here: every step runs in the library's CUDA kernels, and if ``libpkv.so`` is
missing the first call raises instead of computing anything another way.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
# the in-tree build; PKV_LIB may name another build of the same library
LIB_PATH = os.environ.get("PKV_LIB") or os.path.join(_PKG, "_build", "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE_TOO_SMALL = -3
PKV_ERR_LAUNCH = -4

FLAG_BAD_PAGE = 0x1
FLAG_BAD_LEN = 0x2
FLAG_BAD_POS = 0x4
FLAG_TIMEOUT = 0x8
FLAG_NO_PAGE = 0x10

# Every symbol include/pkv.h declares.
EXPORTS = (
    "pkv_split_chunk", "pkv_workspace_bytes", "pkv_workspace_layout", "pkv_plan",
    "pkv_workspace_init", "pkv_rope_table", "paged_kv_append", "paged_decode_attn",
    "paged_decode_step", "paged_decode_partials", "decode_combine", "pkv_status_str",
    "pkv_version", "paged_decode_attn_noalloc", "paged_kv_advance", "decode_attn_contig",
    "paged_prefill_attn", "paged_kv_extend", "paged_decode_step_advance",
    "pkv_testing_set_handoff_wait_ns", "paged_decode_plan", "paged_decode_attn_planned",
    "paged_decode_step_planned", "decode_attn_contig_planned", "paged_prefill_attn_ws",
    "pkv_prefill_workspace_bytes", "pkv_prefill_plan",
)


class PkvError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {msg} ({code})")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int),
        ("num_indices", ctypes.c_int), ("max_seq_len", ctypes.c_int),
        ("scale", ctypes.c_float),
    ]

    def __repr__(self):
        return "Dims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


_lock = threading.Lock()
_lib = None


def lib():
    """Load libpkv.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libpkv.so not found at {LIB_PATH}; build it with "
                "`python -m paged_kv_gqa_16_gb300.build` (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        DP = ctypes.POINTER(Dims)
        sig = {
            "pkv_split_chunk": (I, [DP, I]),
            "pkv_workspace_bytes": (Z, [DP, I]),
            "pkv_workspace_layout": (I, [DP, I, ctypes.POINTER(Z), ctypes.POINTER(Z)]),
            "pkv_plan": (I, [DP, I, ctypes.POINTER(I), ctypes.POINTER(Z)]),
            "pkv_workspace_init": (I, [P, Z, P]),
            "pkv_rope_table": (I, [P, I, I, ctypes.c_double, P]),
            "paged_kv_append": (I, [DP, P, P, P, P, P, P, P, P, P, I, I, P, P]),
            "paged_decode_attn": (I, [DP, P, P, P, P, P, P, I, P, Z, P, P]),
            "paged_decode_step": (I, [DP, P, P, P, P, P, P, P, P, P, I, I, P, Z, P, P]),
            "paged_decode_plan": (I, [DP, P, P, P, I, P, Z, P]),
            "paged_decode_attn_planned": (I, [DP, P, P, P, P, P, P, I, P, Z, P, P]),
            "paged_decode_step_planned": (I, [DP, P, P, P, P, P, P, P, P, P, I, I, P, Z, P, P]),
            "paged_decode_partials": (I, [DP, P, P, P, P, P, P, I, P, Z, P]),
            "decode_combine": (I, [DP, P, P, I, P, P]),
            "paged_decode_attn_noalloc": (I, [DP, P, P, P, P, P, P, I, P, P, P]),
            "paged_kv_advance": (I, [DP, P, P, P, P, I, P, P, P]),
            "paged_decode_step_advance": (I, [DP, P, P, P, P, P, P, P, P, P, I, I, P, Z, P,
                                              P, I, P, P]),
            "decode_attn_contig": (I, [DP, P, P, P, P, P, P, P, P, I, I, P, Z, P, P]),
            "decode_attn_contig_planned": (I, [DP, P, P, P, P, P, P, P, P, I, I, P, Z, P, P]),
            "paged_prefill_attn": (I, [DP, P, P, I, I, P, P, P, P, P, P, P, P]),
            "paged_prefill_attn_ws": (I, [DP, P, P, I, I, P, P, P, P, P, P, Z, P, P, P]),
            "pkv_prefill_workspace_bytes": (Z, [I, I]),
            "pkv_prefill_plan": (I, [DP, I, I, Z, P]),
            "paged_kv_extend": (I, [DP, P, P, P, P, I, P, P, P, P, P, P, I, I, P, P]),
            "pkv_testing_set_handoff_wait_ns": (I, [ctypes.c_ulonglong]),
            "pkv_status_str": (ctypes.c_char_p, [I]),
            "pkv_version": (I, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
        return L


def status_str(code: int) -> str:
    return lib().pkv_status_str(int(code)).decode()


def _check(fn: str, code: int) -> None:
    if code != PKV_OK:
        raise PkvError(fn, code, status_str(code))


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensors passed to libpkv must be contiguous")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dims(B: int, Hq: int, Hkv: int, D: int, page_size: int, num_pages: int,
         num_indices: int, max_seq_len: int, scale: Optional[float] = None) -> Dims:
    return Dims(B, Hq, Hkv, D, page_size, num_pages, num_indices, max_seq_len,
                1.0 / math.sqrt(D) if scale is None else scale)


def version() -> int:
    return lib().pkv_version()


def split_chunk(d: Dims, num_splits: int) -> int:
    return lib().pkv_split_chunk(ctypes.byref(d), num_splits)


def workspace_bytes(d: Dims, num_splits: int) -> int:
    return lib().pkv_workspace_bytes(ctypes.byref(d), num_splits)


def workspace_layout(d: Dims, num_splits: int):
    ml, o = ctypes.c_size_t(), ctypes.c_size_t()
    _check("pkv_workspace_layout",
           lib().pkv_workspace_layout(ctypes.byref(d), num_splits, ctypes.byref(ml),
                                      ctypes.byref(o)))
    return ml.value, o.value


def plan(d: Dims, num_sms: Optional[int] = None):
    if num_sms is None:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    s, ws = ctypes.c_int(), ctypes.c_size_t()
    _check("pkv_plan", lib().pkv_plan(ctypes.byref(d), num_sms, ctypes.byref(s), ctypes.byref(ws)))
    return s.value, ws.value


def workspace_init(workspace, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pkv_workspace_init",
           lib().pkv_workspace_init(_ptr(workspace), ws_bytes, _stream(stream)))


def rope_table(cos_sin, max_pos: int, D: int, base: float, stream=None) -> None:
    _check("pkv_rope_table",
           lib().pkv_rope_table(_ptr(cos_sin), max_pos, D, base, _stream(stream)))


def paged_kv_append(d: Dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                    seq_lens, rope_cos_sin=None, rope_max_pos: int = 0, rope_q: bool = False,
                    status=None, stream=None) -> None:
    _check("paged_kv_append", lib().paged_kv_append(
        ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
        _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), _ptr(rope_cos_sin),
        rope_max_pos, int(bool(rope_q)), _ptr(status), _stream(stream)))


def paged_decode_attn(d: Dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                      num_splits: int, workspace, out, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_decode_attn", lib().paged_decode_attn(
        ctypes.byref(d), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices),
        _ptr(kv_indptr), _ptr(seq_lens), num_splits, _ptr(workspace), ws_bytes, _ptr(out),
        _stream(stream)))


def paged_decode_step(d: Dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                      seq_lens, rope_cos_sin, rope_max_pos: int, num_splits: int, workspace,
                      out, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_decode_step", lib().paged_decode_step(
        ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
        _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), _ptr(rope_cos_sin), rope_max_pos,
        num_splits, _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))


def paged_decode_plan(d: Dims, kv_indices, kv_indptr, seq_lens, num_splits: int, workspace,
                      stream=None) -> None:
    """The step's plan (the block partition and first page-table windows)
    written into the workspace for the *_planned calls of the same step."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_decode_plan", lib().paged_decode_plan(
        ctypes.byref(d), _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), num_splits,
        _ptr(workspace), ws_bytes, _stream(stream)))


def paged_decode_attn_planned(d: Dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                              num_splits: int, workspace, out, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_decode_attn_planned", lib().paged_decode_attn_planned(
        ctypes.byref(d), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices),
        _ptr(kv_indptr), _ptr(seq_lens), num_splits, _ptr(workspace), ws_bytes, _ptr(out),
        _stream(stream)))


def paged_decode_step_planned(d: Dims, q, k_new, v_new, k_pool, v_pool, kv_indices, kv_indptr,
                              seq_lens, rope_cos_sin, rope_max_pos: int, num_splits: int,
                              workspace, out, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_decode_step_planned", lib().paged_decode_step_planned(
        ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
        _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), _ptr(rope_cos_sin), rope_max_pos,
        num_splits, _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))


def paged_kv_advance(d: Dims, seq_lens, kv_indptr, kv_indices, free_pages, free_head,
                     status=None, stream=None) -> None:
    """One more token for every row with seq_lens > 0, and a page from
    free_pages (starting at free_head[0]) for each row whose new token starts
    a page; seq_lens, kv_indices and free_head are updated on the device."""
    num_free = 0 if free_pages is None else int(free_pages.numel())
    _check("paged_kv_advance", lib().paged_kv_advance(
        ctypes.byref(d), _ptr(seq_lens), _ptr(kv_indptr), _ptr(kv_indices), _ptr(free_pages),
        num_free, _ptr(free_head), _ptr(status), _stream(stream)))


def paged_decode_step_advance(d: Dims, q, k_new, v_new, k_pool, v_pool, kv_indices,
                              kv_indptr, seq_lens, rope_cos_sin, rope_max_pos: int,
                              num_splits: int, workspace, out, free_pages, free_head,
                              stream=None) -> None:
    """paged_decode_step, then paged_kv_advance (its flags in the workspace
    status word): one decode-loop step that leaves the metadata ready for
    the next."""
    ws_bytes = workspace.numel() * workspace.element_size()
    num_free = 0 if free_pages is None else int(free_pages.numel())
    _check("paged_decode_step_advance", lib().paged_decode_step_advance(
        ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
        _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), _ptr(rope_cos_sin), rope_max_pos,
        num_splits, _ptr(workspace), ws_bytes, _ptr(out), _ptr(free_pages), num_free,
        _ptr(free_head), _stream(stream)))


def decode_attn_contig(d: Dims, q, k_cache, v_cache, seq_lens, num_splits: int, workspace,
                       out, cache_batch_idx=None, k_new=None, v_new=None, rope_cos_sin=None,
                       rope_max_pos: int = 0, stream=None, planned: bool = False) -> None:
    """Decode over a contiguous cache [num_slots, cache_len, Hkv, D] (d.page_size =
    cache_len, d.num_pages = num_slots); row b reads slot cache_batch_idx[b]
    (None: slot b).  With k_new / v_new it is the whole decode step.
    planned: decode_attn_contig_planned (the table and plan the step's first
    call left in the workspace)."""
    ws_bytes = workspace.numel() * workspace.element_size()
    name = "decode_attn_contig_planned" if planned else "decode_attn_contig"
    _check(name, getattr(lib(), name)(
        ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(cache_batch_idx), _ptr(seq_lens), _ptr(rope_cos_sin), rope_max_pos, num_splits,
        _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))


def paged_prefill_attn(d: Dims, q, qo_indptr, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                       out, status=None, max_q_len: Optional[int] = None, stream=None,
                       workspace=None) -> None:
    """Ragged prefill / extend: q [total_q, Hq, D], row b's chunk the last
    q_len of its seq_lens[b] tokens, each query attending causally.
    max_q_len (>= every chunk length) sizes the grid; None: total_q, always
    safe but many rows then launch many blocks that exit at once -- pass the
    real maximum when it is known.  workspace (a device tensor of
    prefill_workspace_bytes, no initialisation needed): paged_prefill_attn_ws,
    which splits the keys of an under-filled last round."""
    total_q = int(q.shape[0])
    mq = total_q if max_q_len is None else int(max_q_len)
    if workspace is None:
        _check("paged_prefill_attn", lib().paged_prefill_attn(
            ctypes.byref(d), _ptr(q), _ptr(qo_indptr), total_q, mq, _ptr(k_pool), _ptr(v_pool),
            _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), _ptr(out), _ptr(status),
            _stream(stream)))
        return
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_prefill_attn_ws", lib().paged_prefill_attn_ws(
        ctypes.byref(d), _ptr(q), _ptr(qo_indptr), total_q, mq, _ptr(k_pool), _ptr(v_pool),
        _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens), _ptr(workspace), ws_bytes,
        _ptr(out), _ptr(status), _stream(stream)))


def prefill_plan(d: Dims, max_q_len: int, num_sms: int, ws_bytes: int = 0) -> dict:
    """pkv_prefill_plan: the list paged_prefill_attn(_ws) would launch."""
    out = (ctypes.c_int32 * 7)()
    _check("pkv_prefill_plan", lib().pkv_prefill_plan(ctypes.byref(d), int(max_q_len),
                                                       int(num_sms), int(ws_bytes),
                                                       ctypes.cast(out, ctypes.c_void_p)))
    keys = ("pairs", "units", "group_rows", "entries", "split", "split_base", "grid")
    return dict(zip(keys, list(out)))


def prefill_workspace_bytes(D: int, num_sms: int) -> int:
    """pkv_prefill_workspace_bytes: a key-split slot for every SM."""
    return int(lib().pkv_prefill_workspace_bytes(int(D), int(num_sms)))


def paged_kv_extend(d: Dims, q, k_new, v_new, qo_indptr, k_pool, v_pool, kv_indices, kv_indptr,
                    seq_lens, rope_cos_sin=None, rope_max_pos: int = 0, rope_q: bool = False,
                    status=None, stream=None) -> None:
    """Write every row's chunk of new tokens (the last q_len of its seq_lens)
    at their slots: K rotated by position, V copied, q rotated if rope_q."""
    total_q = int(k_new.shape[0])
    _check("paged_kv_extend", lib().paged_kv_extend(
        ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(qo_indptr), total_q,
        _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices), _ptr(kv_indptr), _ptr(seq_lens),
        _ptr(rope_cos_sin), rope_max_pos, int(bool(rope_q)), _ptr(status), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_decode_attn_noalloc(d: Dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                              num_splits: int, out, status=None, stream=None) -> None:
    """paged_decode_attn for callers that cannot allocate: the workspace is
    the library's own 16 MiB device array, shared by every call (calls that
    overlap on the GPU race)."""
    _check("paged_decode_attn_noalloc", lib().paged_decode_attn_noalloc(
        ctypes.byref(d), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices),
        _ptr(kv_indptr), _ptr(seq_lens), num_splits, _ptr(out), _ptr(status),
        _stream(stream)))


def paged_decode_partials(d: Dims, q, k_pool, v_pool, kv_indices, kv_indptr, seq_lens,
                          num_splits: int, workspace, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("paged_decode_partials", lib().paged_decode_partials(
        ctypes.byref(d), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indices),
        _ptr(kv_indptr), _ptr(seq_lens), num_splits, _ptr(workspace), ws_bytes,
        _stream(stream)))


def decode_combine(d: Dims, o_part, ml_part, num_splits: int, out, stream=None) -> None:
    _check("decode_combine", lib().decode_combine(
        ctypes.byref(d), _ptr(o_part), _ptr(ml_part), num_splits, _ptr(out), _stream(stream)))


# ---- conveniences over a caller-owned workspace tensor ----------------------
def alloc_workspace(d: Dims, num_splits: int, device):
    """A uint8 workspace tensor of the right size (torch allocates it once;
    the library itself never allocates).  The status word is zeroed."""
    import torch
    ws = torch.empty(workspace_bytes(d, num_splits) + 256, dtype=torch.uint8, device=device)
    # align the start to 256 bytes
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + workspace_bytes(d, num_splits)]
    workspace_init(ws)
    return ws


def partial_views(d: Dims, num_splits: int, workspace):
    """(o_part [B,Hq,S,D], ml_part [B,Hq,S,2]) fp32 views into a workspace."""
    import torch
    ml_off, o_off = workspace_layout(d, num_splits)
    n = d.B * d.Hq * num_splits
    ml = workspace[ml_off:ml_off + n * 8].view(torch.float32).view(d.B, d.Hq, num_splits, 2)
    o = workspace[o_off:o_off + n * d.D * 4].view(torch.float32).view(d.B, d.Hq, num_splits, d.D)
    return o, ml


def status_word(workspace) -> int:
    """Read the device status word (synchronises through the copy)."""
    import torch
    return int(workspace[:4].view(torch.int32).item()) & 0xFFFFFFFF


DEFAULT_HANDOFF_WAIT_NS = 2_000_000_000


def testing_set_handoff_wait_ns(ns: int) -> None:
    """Test-only: the time limit of the decode kernel's producer/consumer
    hand-off waits (default DEFAULT_HANDOFF_WAIT_NS)."""
    _check("pkv_testing_set_handoff_wait_ns", lib().pkv_testing_set_handoff_wait_ns(int(ns)))
