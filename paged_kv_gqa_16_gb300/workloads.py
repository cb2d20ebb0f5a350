"""Seeded synthetic workloads for paged GQA decode attention.

This module only draws inputs: sequence lengths, page tables and bf16 values.
It holds none of the attention, RoPE or softmax arithmetic, and it is the one
module that both the fp64 oracle (through the tests) and the CUDA library see,
so both get bit-identical inputs.

Every workload follows the shapes of the five decode cases the attention work
targets (GQA decode over a paged pool ``[num_pages, page_size, Hkv, D]``,
packed queries ``[B, Hq, D]``).  Values are N(0, 1) rounded to bf16 by torch;
all randomness comes from one ``torch.Generator`` seeded per workload.

Layout facts a workload fixes (the reading of the pages the library adopts):

* ``seq_lens[b]`` counts the row's tokens INCLUDING the token appended this
  step; the new token's logical position is ``seq_lens[b] - 1``.
* ``kv_indptr`` (``[B+1]``) delimits each row's slice of ``kv_indices``; the
  slice lists the row's pages in logical order, ``ceil(seq_lens[b] /
  page_size)`` of them.
* Pool pages that no row references, slots past a row's end, and the slot the
  new token will occupy are filled with NaN, so a stray read shows up in the
  output.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

NAN_BF16_BITS = 0x7FC0


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    max_seq_len: int          # bound on seq_lens that sizes the split grid
    seq_lens: torch.Tensor    # int32 [B]
    kv_indptr: torch.Tensor   # int32 [B+1]
    kv_indices: torch.Tensor  # int32 [n_ref] physical page ids
    q: torch.Tensor           # bf16 [B, Hq, D]
    k_new: torch.Tensor       # bf16 [B, Hkv, D]
    v_new: torch.Tensor       # bf16 [B, Hkv, D]
    k_pages: torch.Tensor     # bf16 [n_ref, ps, Hkv, D], contents of the referenced pages
    v_pages: torch.Tensor
    rope_base: Optional[float] = 10000.0
    seed: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def n_rep(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def rope_max_pos(self) -> int:
        return max(1, self.max_seq_len)

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    def kv_bytes(self) -> int:
        """Bytes of K and V the attention must read: every token of every row,
        every kv head, K and V, bf16."""
        return self.total_tokens * self.Hkv * self.D * 2 * 2

    # ---- host views (numpy bit patterns) for the oracle -------------------
    def compact_host(self):
        """(k_pool, v_pool, kv_indices) over ONLY the referenced pages: page j
        of the compact pool is physical page kv_indices[j], so the compact
        table is 0..n_ref-1.  Same logical rows as the full pool."""
        kp = self.k_pages.view(torch.int16).numpy().view(np.uint16)
        vp = self.v_pages.view(torch.int16).numpy().view(np.uint16)
        idx = np.arange(self.kv_indices.numel(), dtype=np.int32)
        return kp, vp, idx

    def full_pool_host(self):
        """Full [num_pages, ps, Hkv, D] pools as uint16 bits (small cases)."""
        shape = (self.num_pages, self.page_size, self.Hkv, self.D)
        kp = np.full(shape, NAN_BF16_BITS, dtype=np.uint16)
        vp = np.full(shape, NAN_BF16_BITS, dtype=np.uint16)
        idx = self.kv_indices.numpy().astype(np.int64)
        kp[idx] = self.k_pages.view(torch.int16).numpy().view(np.uint16)
        vp[idx] = self.v_pages.view(torch.int16).numpy().view(np.uint16)
        return kp, vp

    def host(self, name: str) -> np.ndarray:
        t = getattr(self, name)
        if t.dtype == torch.bfloat16:
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        return t.contiguous().numpy()

    # ---- device placement --------------------------------------------------
    def to_device(self, device, pool_pages: Optional[int] = None) -> dict:
        """Device tensors: the full NaN-filled pools with the referenced pages
        placed at their physical ids, plus q, new K/V and the tables."""
        P = self.num_pages if pool_pages is None else pool_pages
        assert P >= self.num_pages
        shape = (P, self.page_size, self.Hkv, self.D)
        k_pool = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=device)
        v_pool = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=device)
        idx = self.kv_indices.to(device=device, dtype=torch.long)
        if idx.numel():
            k_pool[idx] = self.k_pages.to(device)
            v_pool[idx] = self.v_pages.to(device)
        return {
            "q": self.q.to(device).contiguous(),
            "k_new": self.k_new.to(device).contiguous(),
            "v_new": self.v_new.to(device).contiguous(),
            "k_pool": k_pool,
            "v_pool": v_pool,
            "kv_indices": self.kv_indices.to(device),
            "kv_indptr": self.kv_indptr.to(device),
            "seq_lens": self.seq_lens.to(device),
        }


# --------------------------------------------------------------------------
def _randn_bf16(shape, gen, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def build(name: str, *, B: int, Hq: int, Hkv: int, D: int, page_size: int,
          seq_lens, num_pages: Optional[int] = None, pool_factor: float = 2.0,
          max_seq_len: Optional[int] = None, q_scale: float = 1.0,
          rope_base: Optional[float] = 10000.0, seed: int = 0,
          gen: Optional[torch.Generator] = None, notes: Optional[dict] = None,
          fill_new_slot: bool = False) -> Workload:
    """Assemble a workload from explicit lengths: draws the page placement
    (distinct pages, uniformly scattered over the pool) and the bf16 values.
    With ``fill_new_slot`` the slot of position L-1 keeps a random value (for
    attention-only cases that skip the append); otherwise it is NaN."""
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in seq_lens]
    assert len(lens) == B and all(x >= 0 for x in lens)
    n_pages_row = [-(-L // page_size) for L in lens]
    indptr = np.zeros(B + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(n_pages_row)
    n_ref = int(indptr[-1])
    if num_pages is None:
        num_pages = max(1, int(math.ceil(n_ref * pool_factor)))
    assert num_pages >= n_ref, "pool smaller than the pages the rows need"
    perm = torch.randperm(num_pages, generator=gen)[:n_ref].to(torch.int32)

    q = _randn_bf16((B, Hq, D), gen, q_scale)
    k_new = _randn_bf16((B, Hkv, D), gen)
    v_new = _randn_bf16((B, Hkv, D), gen)
    k_pages = _randn_bf16((n_ref, page_size, Hkv, D), gen)
    v_pages = _randn_bf16((n_ref, page_size, Hkv, D), gen)
    # NaN from the new token's slot to the end of each row's last page.
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        first = int(indptr[b])
        for t in range(L if fill_new_slot else L - 1, n_pages_row[b] * page_size):
            pj, sl = divmod(t, page_size)
            k_pages[first + pj, sl] = nan
            v_pages[first + pj, sl] = nan

    return Workload(
        name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=page_size,
        num_pages=num_pages,
        max_seq_len=max(lens + [1]) if max_seq_len is None else max_seq_len,
        seq_lens=torch.tensor(lens, dtype=torch.int32),
        kv_indptr=torch.from_numpy(indptr.astype(np.int32)),
        kv_indices=perm.contiguous(),
        q=q, k_new=k_new, v_new=v_new, k_pages=k_pages, v_pages=v_pages,
        rope_base=rope_base, seed=seed, notes=dict(notes or {}),
    )


# ------------------------------------------------------------ the five cases
def tiny(seed: int = 0) -> Workload:
    """B=2, Hq=4, Hkv=2, D=64, page_size=16, seq_lens {37, 100}; a 16-page
    pool whose pages are handed out in a random permutation."""
    return build("tiny", B=2, Hq=4, Hkv=2, D=64, page_size=16, seq_lens=[37, 100],
                 num_pages=16, seed=seed)


def gqa_1b(seed: int = 0) -> Workload:
    """1B-class GQA decode: B=8, Hq=32, Hkv=8, D=64, page_size=16.  Each row
    holds a 512-token prompt plus 0..512 decoded tokens, uniform, and this
    step appends one more token (RoPE base 10000): seq_len = 512 + U{0..512}
    + 1.  The pool has twice the pages needed, shuffled."""
    gen = torch.Generator().manual_seed(seed)
    lens = (512 + torch.randint(0, 513, (8,), generator=gen) + 1).tolist()
    return build("gqa_1b", B=8, Hq=32, Hkv=8, D=64, page_size=16, seq_lens=lens,
                 pool_factor=2.0, max_seq_len=1025, seed=seed, gen=gen)


def ragged_b32(seed: int = 0, num_pages: int = 65536) -> Workload:
    """Batched ragged decode: B=32, Hq=32, Hkv=8, D=128, page_size=16,
    seq_lens uniform in [512, 4096], pages scattered over a 65536-page pool."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(512, 4097, (32,), generator=gen).tolist()
    return build("ragged_b32", B=32, Hq=32, Hkv=8, D=128, page_size=16,
                 seq_lens=lens, num_pages=num_pages, max_seq_len=4096, seed=seed,
                 gen=gen)


def long_32k(seed: int = 0) -> Workload:
    """Long-context split-KV: B=1, Hq=32, Hkv=8, D=128, page_size=16,
    seq_len 32768 (2048 pages in a shuffled 4096-page pool); q is 2 * N(0,1)
    before rounding, to sharpen the softmax."""
    return build("long_32k", B=1, Hq=32, Hkv=8, D=128, page_size=16,
                 seq_lens=[32768], num_pages=4096, max_seq_len=32768, q_scale=2.0,
                 seed=seed)


SERVING_CAPACITY = 8192


def serving(B: int, seed: int = 0) -> Workload:
    """Serving mix at power-of-two batch B (1..128): Hq=64, Hkv=8, D=128,
    page_size=16.  Live rows: max(1, ceil(3B/4)); their lengths are
    round(lognormal(ln 1024, 1.0)) clipped to [16, 8192]; the remaining rows
    pad the batch with seq_len 0.  The split grid is sized for the 8192-token
    capacity, as a captured graph must be."""
    assert B >= 1 and (B & (B - 1)) == 0
    gen = torch.Generator().manual_seed(seed * 1000 + B)
    live = max(1, -(-3 * B // 4))
    z = torch.randn(live, generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(1024.0) + 1.0 * z).round().clamp(16, SERVING_CAPACITY)
    lens = [int(x) for x in lens.tolist()] + [0] * (B - live)
    return build(f"serving_b{B}", B=B, Hq=64, Hkv=8, D=128, page_size=16,
                 seq_lens=lens, pool_factor=2.0, max_seq_len=SERVING_CAPACITY,
                 seed=seed, gen=gen, notes={"live_rows": live})


SERVING_BATCHES = (1, 2, 4, 8, 16, 32, 64, 128)

CASES = {
    "tiny": tiny,
    "gqa_1b": gqa_1b,
    "ragged_b32": ragged_b32,
    "long_32k": long_32k,
}


def ragged_b32_ps1(seed: int = 0, num_pages: int = 65536 * 16) -> Workload:
    """The ragged B=32 rows in the token-granular layout: page_size 1, every
    token's slot drawn at random from a pool of the same 1,048,576 token
    slots (the reference's req_to_token table is this case)."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(512, 4097, (32,), generator=gen).tolist()
    return build("ragged_b32_ps1", B=32, Hq=32, Hkv=8, D=128, page_size=1,
                 seq_lens=lens, num_pages=num_pages, max_seq_len=4096, seed=seed, gen=gen)


def make(name: str, seed: int = 0, **kw) -> Workload:
    if name == "ragged_b32_ps1":
        return ragged_b32_ps1(seed=seed, **kw)
    if name.startswith("serving_b"):
        return serving(int(name[len("serving_b"):]), seed=seed)
    return CASES[name](seed=seed, **kw)


# ------------------------------------------------------- multi-step decode loop
@dataclass
class LoopState:
    """Inputs of a decode loop whose page table grows on the device.

    Row b owns ``kv_indices[kv_indptr[b] : kv_indptr[b+1]]`` (``cap`` entries,
    a strided table); its first ``ceil(seq_lens[b] / page_size)`` entries are
    the pages it holds, the rest are -1.  ``free_pages`` lists every pool page
    no row holds, shuffled.  ``seq_lens`` are the tokens already cached, before
    the first step; rows with 0 are idle.  Step s appends ``k_new[s]`` /
    ``v_new[s]``.  All bf16 arrays are uint16 bit patterns; pool pages that no
    row holds, and slots past each row's tokens, are NaN."""
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    cap: int
    max_seq_len: int
    steps: int
    seq_lens: np.ndarray      # int32 [B]
    kv_indptr: np.ndarray     # int32 [B+1]
    kv_indices: np.ndarray    # int32 [B*cap]
    free_pages: np.ndarray    # int32 [n_free]
    q: np.ndarray             # uint16 [B, Hq, D]
    k_new: np.ndarray         # uint16 [steps, B, Hkv, D]
    v_new: np.ndarray
    k_pool: np.ndarray        # uint16 [num_pages, page_size, Hkv, D]
    v_pool: np.ndarray
    rope_base: float = 10000.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def decode_loop(*, B: int, Hq: int, Hkv: int, D: int, page_size: int, seq_lens, steps: int,
                cap: int, num_pages: int, seed: int = 0) -> LoopState:
    gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in seq_lens]
    assert len(lens) == B
    held = [-(-L // page_size) for L in lens]
    assert all(h + -(-steps // page_size) + 1 <= cap for h in held), "cap too small"
    n_held = sum(held)
    assert n_held <= num_pages
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32).numpy()
    indptr = (np.arange(B + 1, dtype=np.int64) * cap).astype(np.int32)
    indices = np.full(B * cap, -1, dtype=np.int32)
    k = 0
    for b in range(B):
        indices[b * cap: b * cap + held[b]] = perm[k: k + held[b]]
        k += held[b]
    free = perm[k:].copy()

    def bits(t: torch.Tensor) -> np.ndarray:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()

    q = bits(_randn_bf16((B, Hq, D), gen))
    k_new = bits(_randn_bf16((steps, B, Hkv, D), gen))
    v_new = bits(_randn_bf16((steps, B, Hkv, D), gen))
    k_pool = np.full((num_pages, page_size, Hkv, D), NAN_BF16_BITS, dtype=np.uint16)
    v_pool = np.full_like(k_pool, NAN_BF16_BITS)
    kv = bits(_randn_bf16((2, max(n_held, 1), page_size, Hkv, D), gen))
    j = 0
    for b in range(B):
        for pj in range(held[b]):
            page = indices[b * cap + pj]
            n = min(page_size, lens[b] - pj * page_size)
            k_pool[page, :n] = kv[0, j, :n]
            v_pool[page, :n] = kv[1, j, :n]
            j += 1
    return LoopState(B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=page_size, num_pages=num_pages,
                     cap=cap, max_seq_len=cap * page_size, steps=steps,
                     seq_lens=np.array(lens, dtype=np.int32), kv_indptr=indptr,
                     kv_indices=indices, free_pages=free, q=q, k_new=k_new, v_new=v_new,
                     k_pool=k_pool, v_pool=v_pool)


# ------------------------------------------------------------ contiguous cache
@dataclass
class ContigCase:
    """A contiguous K/V cache [num_slots, cache_len, Hkv, D]; row b reads slot
    ``idx[b]`` over ``seq_lens[b]`` tokens (the new token's slot, position
    seq_len - 1, and everything after it is NaN).  uint16 bf16 bits."""
    B: int
    Hq: int
    Hkv: int
    D: int
    cache_len: int
    num_slots: int
    seq_lens: np.ndarray      # int32 [B]
    idx: np.ndarray           # int32 [B]
    q: np.ndarray             # [B, Hq, D]
    k_new: np.ndarray         # [B, Hkv, D]
    v_new: np.ndarray
    k_cache: np.ndarray       # [num_slots, cache_len, Hkv, D]
    v_cache: np.ndarray
    rope_base: float = 10000.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def contig(*, Hq: int, Hkv: int, D: int, cache_len: int, num_slots: int, seq_lens, idx,
           seed: int = 0, fill_new_slot: bool = False) -> ContigCase:
    gen = torch.Generator().manual_seed(seed)
    lens = np.asarray(seq_lens, dtype=np.int32)
    idx = np.asarray(idx, dtype=np.int32)
    B = len(lens)

    def bits(t: torch.Tensor) -> np.ndarray:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()

    q = bits(_randn_bf16((B, Hq, D), gen))
    k_new = bits(_randn_bf16((B, Hkv, D), gen))
    v_new = bits(_randn_bf16((B, Hkv, D), gen))
    k_cache = bits(_randn_bf16((num_slots, cache_len, Hkv, D), gen))
    v_cache = bits(_randn_bf16((num_slots, cache_len, Hkv, D), gen))
    longest = {}
    for b in range(B):
        longest[int(idx[b])] = max(longest.get(int(idx[b]), 0), int(lens[b]))
    for s, L in longest.items():
        start = L if fill_new_slot else max(L - 1, 0)
        k_cache[s, start:] = NAN_BF16_BITS
        v_cache[s, start:] = NAN_BF16_BITS
    return ContigCase(B=B, Hq=Hq, Hkv=Hkv, D=D, cache_len=cache_len, num_slots=num_slots,
                      seq_lens=lens, idx=idx, q=q, k_new=k_new, v_new=v_new, k_cache=k_cache,
                      v_cache=v_cache)


# ----------------------------------------------------------- prefill / extend
@dataclass
class PrefillCase:
    """A ragged prefill/extend batch over a paged pool: row b's q_lens[b]
    queries are the last q_lens[b] of its seq_lens[b] tokens (their K/V are
    already in the pool).  ``w`` holds the pool, page table and lengths (every
    one of a row's tokens valid); ``q`` [total_q, Hq, D] bf16, ``qo_indptr``
    [B+1] int32 (prefix sum of q_lens)."""
    w: Workload
    q: torch.Tensor
    qo_indptr: torch.Tensor

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    def flops(self) -> int:
        """2 D (q.k) + 2 D (p.v) per (query, head, attended key)."""
        total = 0
        ql = (self.qo_indptr[1:] - self.qo_indptr[:-1]).tolist()
        for L, n in zip(self.w.seq_lens.tolist(), ql):
            first = L - n + 1                     # keys seen by the first query
            total += (first + L) * n // 2
        return 4 * self.w.D * self.w.Hq * total


def prefill(name: str, *, B: int, Hq: int, Hkv: int, D: int, page_size: int, seq_lens,
            q_lens, seed: int = 0, num_pages: Optional[int] = None,
            max_seq_len: Optional[int] = None) -> PrefillCase:
    lens = [int(x) for x in seq_lens]
    ql = [int(x) for x in q_lens]
    assert len(ql) == B and all(0 <= n <= L for n, L in zip(ql, lens))
    gen = torch.Generator().manual_seed(seed)
    w = build(name, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=page_size, seq_lens=lens,
              num_pages=num_pages, max_seq_len=max_seq_len, seed=seed, gen=gen,
              fill_new_slot=True)
    indptr = np.zeros(B + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(ql)
    q = _randn_bf16((int(indptr[-1]), Hq, D), gen)
    return PrefillCase(w=w, q=q, qo_indptr=torch.from_numpy(indptr))


# Prefill / extend shapes the benchmark times: the pages' 512-token prompts at
# the 1B-class head shape, a long prefill, and an extend of 256 new tokens on
# 2,048-token rows.  name -> (label, arguments of prefill()).
PREFILL_SHAPES = {
    "prefill_b32_512": ("prefill B=32 x 512 (Hq 32, Hkv 8, D 64)",
                        dict(B=32, Hq=32, Hkv=8, D=64, page_size=16, seq_lens=[512] * 32,
                             q_lens=[512] * 32)),
    "prefill_b4_4096": ("prefill B=4 x 4096 (Hq 32, Hkv 8, D 128)",
                        dict(B=4, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=[4096] * 4,
                             q_lens=[4096] * 4)),
    "extend_b16": ("extend B=16, 256 new of 2048 (Hq 32, Hkv 8, D 128)",
                   dict(B=16, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=[2048] * 16,
                        q_lens=[256] * 16)),
}


def prefill_shape(name: str, seed: int = 0) -> PrefillCase:
    """The named benchmark prefill shape, seeded."""
    return prefill(name, seed=seed, **PREFILL_SHAPES[name][1])

