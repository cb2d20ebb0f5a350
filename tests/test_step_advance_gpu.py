"""paged_decode_step_advance against the two calls it stands for: a loop of
one paged_kv_advance followed by K step-advances must leave exactly what K
rounds of (paged_kv_advance, paged_decode_step) plus one more advance leave
-- outputs, pools, lengths, page table, free-list head and status word, bit
for bit.  Covered: the persistent path with the advance inside the piece
combine (num_splits > 1), the persistent path with one split (separate
advance launch), the per-(split, kv head, row) path (more rows x kv-head
groups than the persistent kernel takes), and a free list that runs out."""

import numpy as np
import pytest
import torch

from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _setup(B, Hq, Hkv, D, ps, steps, seed, free_keep=None):
    g = torch.Generator().manual_seed(300 + seed)
    lens = torch.randint(1, 3 * ps, (B,), generator=g).tolist()
    lens[0] = 0                                               # an idle row
    if B > 2:
        lens[1], lens[2] = ps, 2 * ps - 1                     # page edges
    held = sum(-(-L // ps) for L in lens)
    need = B * (-(-steps // ps) + 1)
    s = wl.decode_loop(B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, seq_lens=lens, steps=steps,
                       cap=-(-3 * ps // ps) + -(-steps // ps) + 2, num_pages=held + need,
                       seed=seed)
    free = s.free_pages if free_keep is None else s.free_pages[:free_keep]
    dev = "cuda"

    def t16(a):
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    st = dict(q=t16(s.q), k_new=t16(s.k_new), v_new=t16(s.v_new), k_pool=t16(s.k_pool),
              v_pool=t16(s.v_pool), sl=torch.from_numpy(s.seq_lens.copy()).to(dev),
              ptr=torch.from_numpy(s.kv_indptr).to(dev),
              ind=torch.from_numpy(s.kv_indices.copy()).to(dev),
              free=torch.from_numpy(np.ascontiguousarray(free)).to(dev),
              head=torch.zeros(1, dtype=torch.int32, device=dev))
    rope = torch.empty(s.max_seq_len, D // 2, 2, dtype=torch.float32, device=dev)
    pkv.rope_table(rope, s.max_seq_len, D, s.rope_base)
    d = pkv.dims(B, Hq, Hkv, D, ps, s.num_pages, len(s.kv_indices), s.max_seq_len, s.scale)
    return s, d, st, rope


def _clone(st):
    return {k: v.clone() for k, v in st.items()}


def _run(d, st, rope, max_len, steps, S, fused, graph):
    ws = pkv.alloc_workspace(d, S, "cuda")
    B, Hq, D = d.B, d.Hq, d.D
    outs = torch.zeros(steps, B, Hq, D, dtype=torch.bfloat16, device="cuda")

    def loop():
        if fused:
            pkv.paged_kv_advance(d, st["sl"], st["ptr"], st["ind"], st["free"], st["head"],
                                 status=ws)
            for i in range(steps):
                pkv.paged_decode_step_advance(
                    d, st["q"], st["k_new"][i], st["v_new"][i], st["k_pool"], st["v_pool"],
                    st["ind"], st["ptr"], st["sl"], rope, max_len, S, ws, outs[i],
                    st["free"], st["head"])
        else:
            for i in range(steps):
                pkv.paged_kv_advance(d, st["sl"], st["ptr"], st["ind"], st["free"],
                                     st["head"], status=ws)
                pkv.paged_decode_step(d, st["q"], st["k_new"][i], st["v_new"][i],
                                      st["k_pool"], st["v_pool"], st["ind"], st["ptr"],
                                      st["sl"], rope, max_len, S, ws, outs[i])
            pkv.paged_kv_advance(d, st["sl"], st["ptr"], st["ind"], st["free"], st["head"],
                                 status=ws)

    if graph:
        start = _clone(st)
        loop()                                 # warm the launch paths outside capture
        torch.cuda.synchronize()
        for k in st:
            st[k].copy_(start[k])
        ws[:4].zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            loop()
        for k in st:
            st[k].copy_(start[k])
        ws[:4].zero_()
        outs.zero_()
        g.replay()
    else:
        loop()
    torch.cuda.synchronize()
    return outs, pkv.status_word(ws)


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("case", ["combine", "one_split", "split_path", "free_runs_out"])
def test_step_advance_equals_step_then_advance(case):
    steps, ps = 20, 16
    if case == "split_path":
        B, Hq, Hkv, D = 4200, 8, 1, 64             # 4200 rows > the persistent kernel's
    else:
        B, Hq, Hkv, D = 40, 32, 8, 128
    keep = 5 if case == "free_runs_out" else None
    s, d, st0, rope = _setup(B, Hq, Hkv, D, ps, steps, seed=len(case), free_keep=keep)
    S, _ = pkv.plan(d)
    if case == "one_split":
        S = 1
    elif case in ("combine", "free_runs_out"):
        assert S > 1
    results = []
    for fused in (False, True):
        st = _clone(st0)
        outs, word = _run(d, st, rope, s.max_seq_len, steps, S, fused,
                          graph=case != "split_path")
        results.append((outs, word, st))
    (o_a, w_a, st_a), (o_b, w_b, st_b) = results
    assert w_a == w_b
    if case == "free_runs_out":
        assert w_a & pkv.FLAG_NO_PAGE
    else:
        assert w_a == 0
    assert np.array_equal(_bits(o_a), _bits(o_b))
    for k in ("sl", "ind", "head"):
        assert torch.equal(st_a[k], st_b[k]), k
    for k in ("k_pool", "v_pool"):
        assert np.array_equal(_bits(st_a[k]), _bits(st_b[k])), k
    # K + 1 advances: every live row grew by steps + 1 unless it was refused
    if case != "free_runs_out":
        grown = st_b["sl"].cpu().numpy() - s.seq_lens
        assert np.array_equal(grown, np.where(s.seq_lens > 0, steps + 1, 0))
