"""paged_kv_advance on the GPU against the oracle's advance (bit-exact
lengths, page-table entries and free-list head; error flags where the oracle
refuses rows), and a decode loop -- advance, then paged_decode_step, step
after step -- captured in one CUDA graph, against the oracle walking the same
loop."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import bits, compare_out
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _advance_case(B, seed):
    """Rows idle, growing inside a page, starting a page, at or past the
    length bound, with and without room in their table; a free list that
    runs out part way."""
    g = torch.Generator().manual_seed(seed)
    ps, max_len = 16, 80
    lens = torch.randint(0, max_len + 6, (B,), generator=g)
    lens[torch.rand(B, generator=g) < 0.3] = 16 * torch.randint(1, 5, (1,), generator=g).item()
    lens[torch.rand(B, generator=g) < 0.1] = 0
    lens = lens.to(torch.int32).numpy()
    held = -(-lens // ps)
    room = held + torch.randint(0, 3, (B,), generator=g).numpy()      # 0..2 spare entries
    ptr = np.zeros(B + 1, np.int32)
    ptr[1:] = np.cumsum(room)
    ind = np.full(int(ptr[-1]), -1, np.int32)
    for b in range(B):
        ind[ptr[b]: ptr[b] + held[b]] = np.arange(held[b]) + 7 * b
    wants = int(sum(1 for L, r, h in zip(lens, room, held)
                    if 0 < L < max_len and L % ps == 0 and L // ps < r))
    free = torch.randperm(50000, generator=g)[: max(1, wants // 2) + 3].to(torch.int32).numpy()
    return lens, ptr, ind, free, 3, ps, max_len


@pytest.mark.parametrize("B,seed", [(300, 0), (3000, 1), (1, 2)])
def test_advance_matches_oracle(B, seed):
    lens, ptr, ind, free, head0, ps, max_len = _advance_case(B, seed)
    want = oracle.advance(lens, ptr, ind, free, head0, ps, max_len)
    d = pkv.dims(B, 8, 8, 64, ps, 50000, len(ind), max_len)
    dev = "cuda"
    sl = torch.from_numpy(lens.copy()).to(dev)
    ind_d = torch.from_numpy(ind.copy()).to(dev)
    head = torch.tensor([head0], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_kv_advance(d, sl, torch.from_numpy(ptr).to(dev), ind_d,
                         torch.from_numpy(free).to(dev), head, status=status)
    torch.cuda.synchronize()
    sl_w, ind_w, head_w, n_len, n_page, n_bad = want
    assert np.array_equal(sl.cpu().numpy(), sl_w)
    assert np.array_equal(ind_d.cpu().numpy(), ind_w)
    assert int(head.item()) == head_w
    st = int(status.item()) & 0xFFFFFFFF
    assert bool(st & pkv.FLAG_BAD_LEN) == (n_len > 0)
    assert bool(st & pkv.FLAG_NO_PAGE) == (n_page > 0)
    assert bool(st & pkv.FLAG_BAD_PAGE) == (n_bad > 0)
    if B >= 300:
        assert n_page > 0 and n_len > 0    # the case exercises both refusals


def _ulp(a, b):
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


@pytest.mark.parametrize("seed", [0, 1])
def test_decode_loop_in_one_graph(seed):
    g = torch.Generator().manual_seed(100 + seed)
    B, Hq, Hkv, D, ps, steps = 24, 16, 4, 64, 16, 24
    lens = torch.randint(1, 200, (B,), generator=g).tolist()
    lens[0], lens[1], lens[2], lens[3] = 0, 16, 47, 48          # idle, page edges
    s = wl.decode_loop(B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, seq_lens=lens, steps=steps,
                       cap=16, num_pages=400, seed=seed)
    dev = "cuda"
    d = pkv.dims(B, Hq, Hkv, D, ps, s.num_pages, len(s.kv_indices), s.max_seq_len, s.scale)
    S, _ = pkv.plan(d)
    ws = pkv.alloc_workspace(d, S, dev)

    def t16(a):
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    q, k_new, v_new = t16(s.q), t16(s.k_new), t16(s.v_new)
    k_pool, v_pool = t16(s.k_pool), t16(s.v_pool)
    sl = torch.from_numpy(s.seq_lens.copy()).to(dev)
    ptr = torch.from_numpy(s.kv_indptr).to(dev)
    ind = torch.from_numpy(s.kv_indices.copy()).to(dev)
    free = torch.from_numpy(s.free_pages).to(dev)
    head = torch.zeros(1, dtype=torch.int32, device=dev)
    rope = torch.empty(s.max_seq_len, D // 2, 2, dtype=torch.float32, device=dev)
    pkv.rope_table(rope, s.max_seq_len, D, s.rope_base)
    outs = torch.empty(steps, B, Hq, D, dtype=torch.bfloat16, device=dev)
    start = {name: t.clone() for name, t in
             dict(sl=sl, ind=ind, head=head, k_pool=k_pool, v_pool=v_pool).items()}

    def loop():
        for st in range(steps):
            pkv.paged_kv_advance(d, sl, ptr, ind, free, head, status=ws)
            pkv.paged_decode_step(d, q, k_new[st], v_new[st], k_pool, v_pool, ind, ptr, sl,
                                  rope, s.max_seq_len, S, ws, outs[st])

    loop()                                    # eager: also warms the launch paths
    torch.cuda.synchronize()
    for name, t in dict(sl=sl, ind=ind, head=head, k_pool=k_pool, v_pool=v_pool).items():
        t.copy_(start[name])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        loop()
    for name, t in dict(sl=sl, ind=ind, head=head, k_pool=k_pool, v_pool=v_pool).items():
        t.copy_(start[name])
    outs.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert pkv.status_word(ws) == 0

    # the oracle walks the same loop
    o_sl, o_ind, o_head = s.seq_lens.copy(), s.kv_indices.copy(), 0
    o_k, o_v = s.k_pool.copy(), s.v_pool.copy()
    for st in range(steps):
        o_sl, o_ind, o_head, n_len, n_page, n_bad = oracle.advance(
            o_sl, s.kv_indptr, o_ind, s.free_pages, o_head, ps, s.max_seq_len)
        assert n_len == n_page == n_bad == 0
        q2, o_k, o_v = oracle.append(s.q, s.k_new[st], s.v_new[st], o_k, o_v, o_ind,
                                     s.kv_indptr, o_sl, rope_base=s.rope_base, rope_q=True)
        want = oracle.decode(q2, o_k, o_v, o_ind, s.kv_indptr, o_sl, s.scale)
        compare_out(outs[st], want)
        assert np.all(bf16_nonzero_rows(outs[st].cpu(), o_sl))
    assert np.array_equal(sl.cpu().numpy(), o_sl)
    assert np.array_equal(ind.cpu().numpy(), o_ind)
    assert int(head.item()) == o_head
    assert np.array_equal(bits(v_pool), o_v)                   # V copied bit for bit
    kb = bits(k_pool)
    nan = (o_k & 0x7FFF) > 0x7F80
    assert np.array_equal((kb & 0x7FFF) > 0x7F80, nan)
    assert _ulp(kb[~nan], o_k[~nan]).max() <= 1                 # K rotated in fp32


def bf16_nonzero_rows(out, seq_lens):
    """Idle rows are exactly zero; live rows are not all zero."""
    o = out.float().abs().sum(dim=(1, 2)).numpy()
    return np.where(np.asarray(seq_lens) > 0, o > 0, o == 0)
