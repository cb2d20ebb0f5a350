"""paged_prefill_attn on the GPU against the fp64 oracle's prefill: ragged
query chunks (full prefills, extends, single tokens, idle rows), GQA ratios
1..16, page sizes 1..256, head dims 64 and 128, several query and key tiles per
row.  The pools hold NaN in every unreferenced page and past every row's
tokens.  Tolerance: max-abs 2e-2, mean-abs 2e-3."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import compare_out
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run(c, status=None, max_q_len=None):
    w = c.w
    t = w.to_device("cuda")
    P = t["k_pool"].shape[0]
    d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, P, int(w.kv_indices.numel()),
                 w.max_seq_len, w.scale)
    out = torch.full((c.total_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    kw = {} if max_q_len is None else {"max_q_len": max_q_len}
    pkv.paged_prefill_attn(d, c.q.cuda(), c.qo_indptr.cuda(), t["k_pool"], t["v_pool"],
                           t["kv_indices"], t["kv_indptr"], t["seq_lens"], out, status=st, **kw)
    torch.cuda.synchronize()
    return out, int(st.item()) & 0xFFFFFFFF, (d, t)


def _want(c):
    w = c.w
    kp, vp, idx = w.compact_host()
    return oracle.prefill(_bits(c.q), c.qo_indptr.numpy(), kp, vp, idx, w.host("kv_indptr"),
                          w.host("seq_lens"), w.scale)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (16, 8, 128), (32, 8, 128), (64, 8, 128),
                                      (12, 4, 64), (48, 8, 64), (16, 1, 64), (48, 3, 128)])
def test_prefill_shapes(Hq, Hkv, D):
    lens = [40, 1, 300, 133, 0, 17, 64, 65]
    qls = [40, 1, 70, 133, 0, 1, 64, 2]
    c = wl.prefill("pfg", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, page_size=16, seq_lens=lens,
                   q_lens=qls, seed=Hq * 7 + Hkv + D)
    out, st, _ = _run(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("ps,D", [(1, 64), (5, 64), (32, 64), (1, 128), (5, 128), (32, 128),
                                  (8, 128), (64, 64), (256, 128)])
def test_prefill_page_sizes(ps, D):
    """Page sizes that are powers of two >= 8 are loaded by TMA (one box per
    page, or 128-row boxes inside a 256-row page); the others (1, 5) by the
    cp.async gather."""
    lens = [100, 7, 250]
    qls = [37, 7, 129]
    c = wl.prefill("pfp", B=3, Hq=16, Hkv=4, D=D, page_size=ps, seq_lens=lens, q_lens=qls,
                   seed=ps + D)
    out, st, _ = _run(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 4, 64), (16, 4, 128), (8, 8, 128)])
def test_prefill_many_tiles(Hq, Hkv, D):
    """Chunks of several query tiles against several key blocks each: pairs
    of tiles, an odd tile count leaving tile A of a pair idle, and the K/V
    rings reused many times."""
    lens = [1000, 700, 513, 129]
    qls = [700, 700, 200, 129]
    c = wl.prefill("pfm", B=4, Hq=Hq, Hkv=Hkv, D=D, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=21 + D + Hq)
    out, st, _ = _run(c)
    assert st == 0
    compare_out(out, _want(c))



@pytest.mark.parametrize("Hq,Hkv,D", [(8, 4, 64), (16, 4, 128)])
def test_prefill_grouped_rows(Hq, Hkv, D):
    """Chunks of at most 4 pairs of query tiles over more row-heads than one
    group: the unit list takes rows in groups of about one round of units,
    the last group partial (160 row-heads, groups of 152 / pairs rows)."""
    rng = np.random.default_rng(11 + D)
    B = 40
    qls = [int(x) for x in rng.integers(1, 129, size=B)]
    lens = [q + int(x) for q, x in zip(qls, rng.integers(0, 200, size=B))]
    c = wl.prefill("pfgr", B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=31 + D)
    # the chunks' true bound: at most 2 pairs of tiles, so the list is grouped
    out, st, _ = _run(c, max_q_len=max(qls))
    assert st == 0
    compare_out(out, _want(c))

def test_prefill_graph_replay_bitwise():
    lens, qls = [300, 90, 33], [120, 90, 1]
    c = wl.prefill("pfr", B=3, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=5)
    eager, _, (d, t) = _run(c)
    q, qo = c.q.cuda(), c.qo_indptr.cuda()
    out = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_prefill_attn(d, q, qo, t["k_pool"], t["v_pool"], t["kv_indices"],
                               t["kv_indptr"], t["seq_lens"], out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_prefill_flags_bad_chunk():
    """A chunk longer than its row is refused with PKV_FLAG_BAD_LEN; the other
    rows are still right."""
    lens, qls = [50, 20, 80], [50, 20, 30]
    c = wl.prefill("pfb", B=3, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=2)
    want = _want(c)
    w = c.w
    w.seq_lens[1] = 10                      # row 1's chunk of 20 now exceeds it
    out, st, _ = _run(c)
    assert st & pkv.FLAG_BAD_LEN
    compare_out(out[:50], want[:50])
    compare_out(out[70:], want[70:])


def test_prefill_max_q_len():
    """The exact max chunk length gives the same bits as the always-safe
    default (total_q); a bound below a chunk's length is flagged."""
    lens, qls = [300, 90, 33], [120, 90, 1]
    c = wl.prefill("pfq", B=3, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=8)
    ref, st, (d, t) = _run(c)
    assert st == 0
    q, qo = c.q.cuda(), c.qo_indptr.cuda()
    out = torch.empty_like(ref)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_prefill_attn(d, q, qo, t["k_pool"], t["v_pool"], t["kv_indices"], t["kv_indptr"],
                           t["seq_lens"], out, status=st2, max_q_len=max(qls))
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    pkv.paged_prefill_attn(d, q, qo, t["k_pool"], t["v_pool"], t["kv_indices"], t["kv_indptr"],
                           t["seq_lens"], out, status=st2, max_q_len=64)
    torch.cuda.synchronize()
    assert int(st2.item()) & pkv.FLAG_BAD_LEN


# ---- the shapes the benchmark times, in its launch configuration ----------
def _sampled_want(c, picks):
    """The oracle's output for the picked queries only.  Query j of row b's
    chunk sits at position p = seq_len - q_len + j and attends to keys 0..p:
    that is the prefill of a row of p + 1 tokens (the same pages) whose chunk
    is its last token, so each pick becomes a one-query row of its own."""
    w = c.w
    kp, vp, idx = w.compact_host()
    ptr = w.kv_indptr.numpy()
    lens = w.seq_lens.numpy()
    qo = c.qo_indptr.numpy()
    sub_idx, sub_ptr, sub_len, rows = [], [0], [], []
    for b, j in picks:
        p = int(lens[b]) - int(qo[b + 1] - qo[b]) + j
        need = -(-(p + 1) // w.page_size)
        sub_idx.extend(idx[ptr[b]:ptr[b] + need].tolist())
        sub_ptr.append(len(sub_idx))
        sub_len.append(p + 1)
        rows.append(int(qo[b]) + j)
    want = oracle.prefill(_bits(c.q)[rows], np.arange(len(picks) + 1, dtype=np.int32), kp, vp,
                          np.array(sub_idx, dtype=np.int32), np.array(sub_ptr, dtype=np.int32),
                          np.array(sub_len, dtype=np.int32), w.scale)
    return rows, want


def _picks(c, runs, n_random, seed):
    """Per row: the query runs given (first and last queries, runs across
    tile and tile-pair boundaries) plus n_random random queries."""
    g = np.random.default_rng(seed)
    qo = c.qo_indptr.numpy()
    out = []
    for b in range(c.w.B):
        n = int(qo[b + 1] - qo[b])
        js = set()
        for a, e in runs:
            js.update(j for j in range(a if a >= 0 else n + a, e if e > 0 else n + e)
                      if 0 <= j < n)
        js.update(g.integers(0, n, n_random).tolist())
        out += [(b, j) for j in sorted(js)]
    return out


def test_prefill_bench_shape_b32_512_full():
    """32 prompts of 512 at D = 64, every query against the oracle."""
    c = wl.prefill_shape("prefill_b32_512")
    out, st, _ = _run_bench_config(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("name,runs,n_random", [
    # 4 rows of 4096: tiles of 32 tokens (n_rep 4), pairs of 64
    ("prefill_b4_4096", [(0, 8), (28, 37), (60, 69), (2040, 2057), (-8, 0)], 24),
    # 16 extends of 256 new tokens on rows of 2048
    ("extend_b16", [(0, 4), (30, 34), (62, 66), (126, 130), (-4, 0)], 4),
])
def test_prefill_bench_shape_sampled(name, runs, n_random):
    """The large bench shapes: the GPU computes every query; the oracle
    checks a sample of them, each as a one-query row of its own."""
    c = wl.prefill_shape(name)
    out, st, _ = _run_bench_config(c)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    rows, want = _sampled_want(c, _picks(c, runs, n_random, seed=len(name)))
    compare_out(out[rows], want)


def _run_bench_config(c):
    """One call as the benchmark makes it: max_q_len is the longest chunk, and
    a workspace with a part slot per SM (paged_prefill_attn_ws)."""
    w = c.w
    t = w.to_device("cuda")
    P = t["k_pool"].shape[0]
    d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, P, int(w.kv_indices.numel()),
                 w.max_seq_len, w.scale)
    out = torch.full((c.total_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ql = (c.qo_indptr[1:] - c.qo_indptr[:-1]).tolist()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ws = torch.zeros(pkv.prefill_workspace_bytes(w.D, sms), dtype=torch.uint8, device="cuda")
    pkv.paged_prefill_attn(d, c.q.cuda(), c.qo_indptr.cuda(), t["k_pool"], t["v_pool"],
                           t["kv_indices"], t["kv_indptr"], t["seq_lens"], out, status=st,
                           max_q_len=max(ql), workspace=ws)
    torch.cuda.synchronize()
    return out.cpu(), int(st.item()) & 0xFFFFFFFF, (d, t)
