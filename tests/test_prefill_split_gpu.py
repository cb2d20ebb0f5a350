"""paged_prefill_attn_ws, the prefill with a key split, on the GPU against the
fp64 oracle's prefill.  The split cuts the units of an under-filled last
round (every unit, when they are few) into parts over consecutive key
blocks; each part leaves its rows (bf16, normalised on its own base) and
their fp32 (base, l) in the workspace and a merge kernel combines them.  Cases: extends and full causal prefills of a few long
rows (the units of many key blocks split, the causal diagonal in a unit's
last part), a list whose last round alone is split, a mix of split and
unsplit units in one round, workspaces with room for fewer parts, a
workspace full of garbage, graph replay, and outputs only 16-byte aligned
(the 16-byte row stores).  Tolerance as for
paged_prefill_attn: max-abs 2e-2, mean-abs 2e-3."""

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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _want(c):
    w = c.w
    kp, vp, idx = w.compact_host()
    return oracle.prefill(_bits(c.q), c.qo_indptr.numpy(), kp, vp, idx, w.host("kv_indptr"),
                          w.host("seq_lens"), w.scale)


def _setup(c):
    w = c.w
    t = w.to_device("cuda")
    d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, t["k_pool"].shape[0],
                 int(w.kv_indices.numel()), w.max_seq_len, w.scale)
    return d, t


def _call(c, d, t, ws, out, st, max_q_len):
    pkv.paged_prefill_attn(d, c.q.cuda(), c.qo_indptr.cuda(), t["k_pool"], t["v_pool"],
                           t["kv_indices"], t["kv_indptr"], t["seq_lens"], out, status=st,
                           max_q_len=max_q_len, workspace=ws)


def _run_ws(c, slots=None, fill=0):
    """One call with a workspace of `slots` part slots (default: one per SM)
    whose bytes all hold `fill`; returns the output, the status and the
    workspace."""
    w = c.w
    d, t = _setup(c)
    n = _sms() if slots is None else slots
    nbytes = pkv.prefill_workspace_bytes(w.D, n)
    assert nbytes > 0
    ws = torch.full((nbytes,), fill, dtype=torch.uint8, device="cuda")
    out = torch.full((c.total_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ql = (c.qo_indptr[1:] - c.qo_indptr[:-1]).tolist()
    _call(c, d, t, ws, out, st, max(ql))
    torch.cuda.synchronize()
    return out, int(st.item()) & 0xFFFFFFFF, ws


@pytest.mark.parametrize("D", [64, 128])
def test_split_extend_few_rows(D):
    """Two extends (256 and 200 new tokens) on rows of about 3,000: 2 rows x 2
    kv heads x 4 pairs = 16 units, each cut into SMs / 16 parts (9 on 152
    SMs) of 2+ blocks."""
    c = wl.prefill("pss", B=2, Hq=8, Hkv=2, D=D, page_size=16, seq_lens=[3000, 2817],
                   q_lens=[256, 200], seed=40 + D)
    out, st, ws = _run_ws(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("D,Hq,Hkv,L", [(64, 8, 2, 1024), (128, 8, 2, 1200),
                                        (128, 16, 1, 1000)])
def test_split_causal_prefill(D, Hq, Hkv, L):
    """A full causal prefill of one row: units from one key block (run whole)
    to L / 128 (split), the causal diagonal in each unit's last part only;
    32-64 units, so 2-4 parts."""
    c = wl.prefill("psc", B=1, Hq=Hq, Hkv=Hkv, D=D, page_size=16, seq_lens=[L], q_lens=[L],
                   seed=50 + D + L)
    out, st, ws = _run_ws(c)
    assert st == 0
    compare_out(out, _want(c))


def test_split_last_round_only():
    """More units than SMs: 21 rows x 8 kv heads, one pair each (168 units),
    so only the last round's units (168 - SMs) are split, into 2-3 parts of
    the rows' 5-7 key blocks."""
    B = 21
    lens = [600 + 13 * b for b in range(B)]
    qls = [64 - (b % 5) for b in range(B)]
    c = wl.prefill("psl", B=B, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=61)
    out, st, ws = _run_ws(c)
    assert st == 0
    compare_out(out, _want(c))


def test_split_mixed_round():
    """One round (7 rows x 2 kv heads x 5 pairs = 70 units) with units of 1-3
    blocks (run whole), units of 4+ blocks (split in two), pairs past a
    row's chunk, a row with no chunk and single-token chunks."""
    lens = [2000, 300, 0, 45, 1200, 9, 2600]
    qls = [130, 300, 0, 1, 64, 9, 1]
    c = wl.prefill("psm", B=len(lens), Hq=8, Hkv=2, D=128, page_size=16, seq_lens=lens,
                   q_lens=qls, seed=71)
    out, st, ws = _run_ws(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("slots", [1, 3, 5])
def test_split_small_workspace(slots):
    """A workspace with room for few parts: 2 units (1 row x 2 kv heads x 1
    pair) get slots // 2 parts each (none below two), the same results."""
    c = wl.prefill("psw", B=1, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[2048],
                   q_lens=[60], seed=81)
    out, st, ws = _run_ws(c, slots=slots)
    assert st == 0
    compare_out(out, _want(c))


def test_split_close_to_whole_units():
    """The split result differs from paged_prefill_attn's by the parts' one
    extra bf16 rounding: both against the oracle, and each other within two
    bf16 steps."""
    c = wl.prefill("psx", B=1, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=[4096],
                   q_lens=[512], seed=91)
    split, st, _ = _run_ws(c)
    assert st == 0
    d, t = _setup(c)
    whole = torch.empty_like(split)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    _call(c, d, t, None, whole, st2, 512)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    want = _want(c)
    compare_out(split, want)
    compare_out(whole, want)
    diff = (split.float() - whole.float()).abs()
    assert diff.max().item() <= 2 ** -6 * max(1.0, whole.float().abs().max().item())
    # the parts' extra rounding shows in some of the 2M outputs: the split ran
    assert not torch.equal(split.view(torch.int16), whole.view(torch.int16))


def test_split_graph_replay_bitwise():
    """Captured in a CUDA graph and replayed twice on one workspace: the same
    bits as the eager call each time (the merge sums parts in part order)."""
    c = wl.prefill("psg", B=2, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[2500, 1900],
                   q_lens=[192, 100], seed=101)
    eager, st, ws = _run_ws(c)
    assert st == 0
    d, t = _setup(c)
    q, qo = c.q.cuda(), c.qo_indptr.cuda()
    out = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_prefill_attn(d, q, qo, t["k_pool"], t["v_pool"], t["kv_indices"],
                               t["kv_indptr"], t["seq_lens"], out, max_q_len=192, workspace=ws)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    

def test_split_garbage_workspace():
    """The workspace needs no initialisation: every byte 0xFF (NaN in both
    the bf16 rows and the fp32 pairs) before the call gives the same bits as
    a zeroed one."""
    c = wl.prefill("psn", B=1, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[2200],
                   q_lens=[100], seed=121)
    a, st, _ = _run_ws(c)
    b, st2, _ = _run_ws(c, fill=255)
    assert st == 0 and st2 == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    compare_out(a, _want(c))


def test_split_rejects_misaligned_workspace():
    c = wl.prefill("psa", B=1, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[300],
                   q_lens=[30], seed=111)
    d, t = _setup(c)
    ws = torch.zeros(pkv.prefill_workspace_bytes(64, _sms()) + 256, dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((c.total_q, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        _call(c, d, t, ws[8:], out, None, 30)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG


def test_split_flags_bad_chunk():
    """A chunk longer than its row is refused (PKV_FLAG_BAD_LEN) in a split
    list too: its parts do nothing, the merge skips it, and the other rows'
    parts (8 and 6 of them) are still right."""
    lens, qls = [2000, 20, 1500], [50, 20, 30]
    c = wl.prefill("psb", B=3, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=lens, q_lens=qls,
                   seed=131)
    want = _want(c)
    c.w.seq_lens[1] = 10                    # row 1's chunk of 20 now exceeds it
    out, st, _ = _run_ws(c)
    assert st & pkv.FLAG_BAD_LEN
    compare_out(out[:50], want[:50])
    compare_out(out[70:], want[70:])


@pytest.mark.parametrize("ps,D", [(5, 64), (1, 128)])
def test_split_gathered_pages(ps, D):
    """Page sizes the TMA path does not take (5, 1): the cp.async gather loads
    each part's blocks from its own first key, and the last part's partial V
    block is zero-filled."""
    c = wl.prefill("psp", B=2, Hq=8, Hkv=2, D=D, page_size=ps, seq_lens=[1700, 1333],
                   q_lens=[100, 77], seed=140 + ps + D)
    out, st, _ = _run_ws(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (12, 4), (48, 3)])
def test_split_gqa_ratios(Hq, Hkv):
    """GQA ratios 1, 3 and 16 in a split list: tiles of 128, 42 (126 rows used)
    and 8 tokens, 8 to 39 units cut 3 to 16 ways."""
    c = wl.prefill("psq", B=1, Hq=Hq, Hkv=Hkv, D=128, page_size=16, seq_lens=[2000],
                   q_lens=[200], seed=150 + Hq + Hkv)
    out, st, _ = _run_ws(c)
    assert st == 0
    compare_out(out, _want(c))


@pytest.mark.parametrize("D,ws", [(64, False), (64, True), (128, False), (128, True)])
def test_out_16_byte_aligned(D, ws):
    """An output 16 but not 32 bytes aligned takes the 16-byte row stores
    (the 32-byte stores need 32): the same values.  With a workspace the
    split parts still store theirs with 32-byte stores, into the workspace."""
    c = wl.prefill("pso", B=2, Hq=12, Hkv=4, D=D, page_size=16, seq_lens=[1500, 700],
                   q_lens=[90, 33], seed=160 + D + ws)
    w = c.w
    d, t = _setup(c)
    n = c.total_q * w.Hq * w.D
    buf = torch.full((n + 64,), float("nan"), dtype=torch.bfloat16, device="cuda")
    off = next(i for i in range(0, 64, 8) if (buf.data_ptr() + 2 * i) % 32 == 16)
    out = buf[off:off + n].view(c.total_q, w.Hq, w.D)
    wsb = (torch.empty(pkv.prefill_workspace_bytes(D, _sms()), dtype=torch.uint8, device="cuda")
           if ws else None)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _call(c, d, t, wsb, out, st, 90)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    compare_out(out, _want(c))
