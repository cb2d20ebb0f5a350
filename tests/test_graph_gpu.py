"""The whole step (append + split decode + combine) captured in a CUDA graph:
replay equals the eager run bit for bit, and stays correct after the
lengths, page tables and inputs are rewritten in place at the same
addresses (the serving case: one graph per power-of-two batch, sized for
an 8192-token capacity)."""

import numpy as np
import pytest
import torch

from gpu_cases import compare_out, oracle_step
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CAP = wl.SERVING_CAPACITY


def _serving_like(B, seed, num_pages):
    src = wl.serving(B, seed=seed)
    return wl.build(f"graph_b{B}_s{seed}", B=B, Hq=64, Hkv=8, D=128, page_size=16,
                    seq_lens=src.seq_lens.tolist(), num_pages=num_pages, max_seq_len=CAP,
                    seed=seed)


class Fixed:
    """Buffers at fixed addresses, sized for the capacity."""

    def __init__(self, B, num_pages):
        dev = "cuda"
        self.B = B
        n_idx = B * (CAP // 16)
        self.d = pkv.dims(B, 64, 8, 128, 16, num_pages, n_idx, CAP)
        self.S, _ = pkv.plan(self.d)
        self.ws = pkv.alloc_workspace(self.d, self.S, dev)
        self.k_pool = torch.full((num_pages, 16, 8, 128), float("nan"), dtype=torch.bfloat16,
                                 device=dev)
        self.v_pool = torch.full_like(self.k_pool, float("nan"))
        self.kv_indices = torch.zeros(n_idx, dtype=torch.int32, device=dev)
        self.kv_indptr = torch.zeros(B + 1, dtype=torch.int32, device=dev)
        self.seq_lens = torch.zeros(B, dtype=torch.int32, device=dev)
        self.q_in = torch.empty(B, 64, 128, dtype=torch.bfloat16, device=dev)
        self.q = torch.empty_like(self.q_in)
        self.k_new = torch.empty(B, 8, 128, dtype=torch.bfloat16, device=dev)
        self.v_new = torch.empty_like(self.k_new)
        self.out = torch.empty(B, 64, 128, dtype=torch.bfloat16, device=dev)
        self.rope = torch.empty(CAP, 64, 2, dtype=torch.float32, device=dev)
        pkv.rope_table(self.rope, CAP, 128, 10000.0)

    def load(self, w):
        t = w.to_device("cuda")
        self.k_pool.copy_(t["k_pool"])
        self.v_pool.copy_(t["v_pool"])
        self.kv_indices.zero_()
        self.kv_indices[: t["kv_indices"].numel()].copy_(t["kv_indices"])
        self.kv_indptr.copy_(t["kv_indptr"])
        self.seq_lens.copy_(t["seq_lens"])
        self.q_in.copy_(t["q"])
        self.k_new.copy_(t["k_new"])
        self.v_new.copy_(t["v_new"])

    def step(self):
        self.q.copy_(self.q_in)
        pkv.paged_kv_append(self.d, self.q, self.k_new, self.v_new, self.k_pool, self.v_pool,
                            self.kv_indices, self.kv_indptr, self.seq_lens,
                            rope_cos_sin=self.rope, rope_max_pos=CAP, rope_q=True,
                            status=self.ws)
        pkv.paged_decode_attn(self.d, self.q, self.k_pool, self.v_pool, self.kv_indices,
                              self.kv_indptr, self.seq_lens, self.S, self.ws, self.out)


@pytest.mark.parametrize("B", [1, 16, 128])
def test_graph_replay_bitwise_and_rebind(B):
    need = max(sum(-(-L // 16) for L in wl.serving(B, seed=s).seq_lens.tolist())
               for s in (0, 1))
    num_pages = 2 * need + 16
    f = Fixed(B, num_pages)
    w1 = _serving_like(B, 0, num_pages)
    w2 = _serving_like(B, 1, num_pages)

    f.load(w1)
    f.step()
    eager1 = f.out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        f.step()
    f.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(f.out.view(torch.int16), eager1.view(torch.int16))
    compare_out(f.out, oracle_step(w1)["out"])

    # new lengths, tables and inputs at the same addresses
    f.load(w2)
    f.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    replay2 = f.out.clone()
    f.step()
    torch.cuda.synchronize()
    assert torch.equal(replay2.view(torch.int16), f.out.view(torch.int16))
    compare_out(replay2, oracle_step(w2)["out"])
    assert pkv.status_word(f.ws) == 0


@pytest.mark.parametrize("B", [4, 64])
def test_graph_fused_step(B):
    """paged_decode_step captured once; replays with rebound inputs equal eager."""
    need = max(sum(-(-L // 16) for L in wl.serving(B, seed=s).seq_lens.tolist())
               for s in (0, 1))
    num_pages = 2 * need + 16
    f = Fixed(B, num_pages)

    def fused():
        pkv.paged_decode_step(f.d, f.q_in, f.k_new, f.v_new, f.k_pool, f.v_pool, f.kv_indices,
                              f.kv_indptr, f.seq_lens, f.rope, CAP, f.S, f.ws, f.out)

    w1, w2 = _serving_like(B, 0, num_pages), _serving_like(B, 1, num_pages)
    f.load(w1)
    fused()
    eager = f.out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fused()
    f.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(f.out.view(torch.int16), eager.view(torch.int16))
    f.load(w2)
    g.replay()
    torch.cuda.synchronize()
    compare_out(f.out, oracle_step(w2)["out"])
    assert pkv.status_word(f.ws) == 0
