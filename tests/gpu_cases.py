"""Helpers shared by the GPU parity tests: run one workload through the fp64
oracle and through libpkv on the same seeded inputs, and compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

# bf16 output vs fp64 oracle (the target's stated tolerance)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def oracle_step(w: wl.Workload, rope_q: bool = True):
    """Oracle append (RoPE on K and, if asked, q) then oracle decode, on the
    compact pool (referenced pages only; same logical rows as the full one)."""
    kp, vp, idx = w.compact_host()
    q2, kp2, vp2 = oracle.append(w.host("q"), w.host("k_new"), w.host("v_new"), kp, vp, idx,
                                 w.host("kv_indptr"), w.host("seq_lens"),
                                 rope_base=w.rope_base, rope_q=rope_q)
    out = oracle.decode(q2, kp2, vp2, idx, w.host("kv_indptr"), w.host("seq_lens"), w.scale)
    return dict(q=q2, k_pages=kp2, v_pages=vp2, idx=idx, out=out)


class GpuCase:
    """Device state of one workload: pools, tables, RoPE table, workspace."""

    def __init__(self, w: wl.Workload, num_splits: int | None = None, device="cuda",
                 pool_pages: int | None = None, max_seq_len: int | None = None):
        self.w = w
        self.t = w.to_device(device, pool_pages=pool_pages)
        P = self.t["k_pool"].shape[0]
        self.d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, P, int(w.kv_indices.numel()),
                          w.max_seq_len if max_seq_len is None else max_seq_len, w.scale)
        if num_splits is None:
            num_splits, _ = pkv.plan(self.d)
        self.S = num_splits
        self.ws = pkv.alloc_workspace(self.d, self.S, device)
        self.rope_max_pos = max(w.max_seq_len, 1)
        self.rope = torch.empty(self.rope_max_pos, w.D // 2, 2, dtype=torch.float32, device=device)
        pkv.rope_table(self.rope, self.rope_max_pos, w.D, w.rope_base or 10000.0)
        self.out = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device=device)

    def append(self, rope_q: bool = True):
        t = self.t
        pkv.paged_kv_append(self.d, t["q"], t["k_new"], t["v_new"], t["k_pool"], t["v_pool"],
                            t["kv_indices"], t["kv_indptr"], t["seq_lens"],
                            rope_cos_sin=self.rope if self.w.rope_base else None,
                            rope_max_pos=self.rope_max_pos, rope_q=rope_q, status=self.ws)

    def decode(self, num_splits: int | None = None):
        t = self.t
        S = self.S if num_splits is None else num_splits
        assert S <= self.S or pkv.workspace_bytes(self.d, S) <= self.ws.numel()
        pkv.paged_decode_attn(self.d, t["q"], t["k_pool"], t["v_pool"], t["kv_indices"],
                              t["kv_indptr"], t["seq_lens"], S, self.ws, self.out)
        return self.out

    def status(self) -> int:
        torch.cuda.synchronize()
        return pkv.status_word(self.ws)


def compare_out(got: torch.Tensor, want: np.ndarray, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    """Element-wise check of a bf16 output against the fp64 oracle.

    Rows (first axis) whose oracle output is exactly zero everywhere are the
    padding rows (seq_len 0: the oracle writes +0.0 and reads nothing).  They
    must be exactly zero on the GPU too, and they are left out of the mean,
    which would otherwise be diluted by their zero error; the max covers
    every element."""
    g = bf16_to_f64(got)
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - want)
    assert err.max() <= max_abs, f"max abs err {err.max():.3e}"
    flat_w = want.reshape(want.shape[0], -1)
    pad = ~np.any(flat_w != 0.0, axis=1)
    if pad.any():
        assert not np.any(g.reshape(g.shape[0], -1)[pad] != 0.0), "padding row not zero"
    live = err.reshape(err.shape[0], -1)[~pad]
    mean = float(live.mean()) if live.size else 0.0
    assert mean <= mean_abs, f"mean abs err over live rows {mean:.3e}"
    return float(err.max()), mean


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits): 2^(e - 7) for
    |x| in [2^e, 2^(e+1)), and the subnormal spacing 2^-133 at the bottom."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(ax > 0, np.exp2(e - 7.0), 2.0 ** -133)


def ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (same-sign finite values)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)
