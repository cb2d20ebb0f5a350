"""decode_attn_contig: decode, and the whole step, over a contiguous K/V cache
[num_slots, cache_len, Hkv, D] read through cache_batch_idx -- against the
oracle on the same cache seen as a pool with one page of cache_len tokens per
row, and bit for bit against paged_decode_attn on the same memory cut into
16-token pages."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import bits, compare_out
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()


def _run(c, S=None, idx=True, step=False):
    d = pkv.dims(c.B, c.Hq, c.Hkv, c.D, c.cache_len, c.num_slots, c.B, c.cache_len, c.scale)
    S = S or pkv.plan(d)[0]
    ws = pkv.alloc_workspace(d, S, "cuda")
    kc, vc = _dev(c.k_cache), _dev(c.v_cache)
    out = torch.empty(c.B, c.Hq, c.D, dtype=torch.bfloat16, device="cuda")
    rope = None
    if step:
        rope = torch.empty(c.cache_len, c.D // 2, 2, dtype=torch.float32, device="cuda")
        pkv.rope_table(rope, c.cache_len, c.D, c.rope_base)
    pkv.decode_attn_contig(d, _dev(c.q), kc, vc, torch.from_numpy(c.seq_lens).cuda(), S, ws, out,
                           cache_batch_idx=torch.from_numpy(c.idx).cuda() if idx else None,
                           k_new=_dev(c.k_new) if step else None,
                           v_new=_dev(c.v_new) if step else None,
                           rope_cos_sin=rope, rope_max_pos=c.cache_len if step else 0)
    torch.cuda.synchronize()
    assert pkv.status_word(ws) == 0
    return out, kc, vc


def _oracle(c, step=False):
    ptr = np.arange(c.B + 1, dtype=np.int32)
    q, kc, vc = c.q, c.k_cache, c.v_cache
    if step:
        q, kc, vc = oracle.append(c.q, c.k_new, c.v_new, kc, vc, c.idx, ptr, c.seq_lens,
                                  rope_base=c.rope_base, rope_q=True)
    return oracle.decode(q, kc, vc, c.idx, ptr, c.seq_lens, c.scale), kc, vc


@pytest.mark.parametrize("S", [None, 1, 5])
def test_contig_decode_matches_oracle(S):
    c = wl.contig(Hq=16, Hkv=4, D=128, cache_len=300, num_slots=6, seq_lens=[1, 300, 0, 157],
                  idx=[5, 0, 3, 3], seed=3, fill_new_slot=True)
    out, _, _ = _run(c, S)
    want, _, _ = _oracle(c)
    compare_out(out, want)
    assert torch.count_nonzero(out[2]) == 0


def test_contig_identity_slots():
    c = wl.contig(Hq=8, Hkv=8, D=64, cache_len=77, num_slots=5, seq_lens=[77, 5, 40, 1, 0],
                  idx=[0, 1, 2, 3, 4], seed=4, fill_new_slot=True)
    out, _, _ = _run(c, idx=False)
    compare_out(out, _oracle(c)[0])


def test_contig_step_matches_oracle():
    c = wl.contig(Hq=32, Hkv=8, D=128, cache_len=512, num_slots=7, seq_lens=[512, 33, 1, 260],
                  idx=[6, 2, 0, 4], seed=5)
    out, kc, vc = _run(c, step=True)
    want, ok, ov = _oracle(c, step=True)
    compare_out(out, want)
    assert np.array_equal(bits(vc), ov)
    kb = bits(kc)
    nan = (ok & 0x7FFF) > 0x7F80
    assert np.array_equal((kb & 0x7FFF) > 0x7F80, nan)
    diff = np.abs(kb[~nan].astype(np.int32) - ok[~nan].astype(np.int32))
    assert diff.max() <= 1


def test_contig_equals_paged_bitwise():
    """The same memory as 16-token pages through paged_decode_attn gives the
    same bits: the partition and the per-token arithmetic do not depend on
    where a token's page starts."""
    c = wl.contig(Hq=32, Hkv=8, D=128, cache_len=320, num_slots=9,
                  seq_lens=[320, 17, 200, 0, 64, 129], idx=[8, 0, 3, 5, 1, 7], seed=6,
                  fill_new_slot=True)
    out_c, kc, vc = _run(c)
    nps = c.cache_len // 16
    lens = c.seq_lens
    pages = [[int(c.idx[b]) * nps + j for j in range(-(-int(L) // 16))] for b, L in enumerate(lens)]
    ptr = np.zeros(c.B + 1, np.int32)
    ptr[1:] = np.cumsum([len(p) for p in pages])
    ind = np.array([x for p in pages for x in p], np.int32)
    d = pkv.dims(c.B, c.Hq, c.Hkv, c.D, 16, c.num_slots * nps, len(ind), c.cache_len, c.scale)
    S = pkv.plan(pkv.dims(c.B, c.Hq, c.Hkv, c.D, c.cache_len, c.num_slots, c.B, c.cache_len,
                          c.scale))[0]
    ws = pkv.alloc_workspace(d, S, "cuda")
    out_p = torch.empty_like(out_c)
    pkv.paged_decode_attn(d, _dev(c.q), kc.view(-1, 16, c.Hkv, c.D), vc.view(-1, 16, c.Hkv, c.D),
                          torch.from_numpy(ind).cuda(), torch.from_numpy(ptr).cuda(),
                          torch.from_numpy(lens).cuda(), S, ws, out_p)
    torch.cuda.synchronize()
    assert torch.equal(out_c.view(torch.int16), out_p.view(torch.int16))


def test_contig_planned_layers_bitwise():
    """A step's later layers: decode_attn_contig_planned reuses the table and
    the plan the first call left in the workspace, launches no table kernel,
    and gives the first call's bits, for the attention and the whole step."""
    c = wl.contig(Hq=32, Hkv=8, D=128, cache_len=512, num_slots=7, seq_lens=[512, 33, 1, 260],
                  idx=[6, 2, 0, 4], seed=9, fill_new_slot=True)
    d = pkv.dims(c.B, c.Hq, c.Hkv, c.D, c.cache_len, c.num_slots, c.B, c.cache_len, c.scale)
    S = pkv.plan(d)[0]
    ws = pkv.alloc_workspace(d, S, "cuda")
    kc, vc = _dev(c.k_cache), _dev(c.v_cache)
    q, lens = _dev(c.q), torch.from_numpy(c.seq_lens).cuda()
    idx = torch.from_numpy(c.idx).cuda()
    outs = [torch.empty(c.B, c.Hq, c.D, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    pkv.decode_attn_contig(d, q, kc, vc, lens, S, ws, outs[0], cache_batch_idx=idx)
    for o in outs[1:]:
        pkv.decode_attn_contig(d, q, kc, vc, lens, S, ws, o, cache_batch_idx=idx, planned=True)
    torch.cuda.synchronize()
    assert pkv.status_word(ws) == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    compare_out(outs[1], _oracle(c)[0])
    # the whole step (the new token written at seq_len - 1 of its slot)
    rope = torch.empty(c.cache_len, c.D // 2, 2, dtype=torch.float32, device="cuda")
    pkv.rope_table(rope, c.cache_len, c.D, c.rope_base)
    kn, vn = _dev(c.k_new), _dev(c.v_new)
    kc2, vc2 = kc.clone(), vc.clone()
    step_outs = []
    for planned, (k_, v_) in ((False, (kc, vc)), (True, (kc2, vc2))):
        o = torch.empty_like(outs[0])
        pkv.decode_attn_contig(d, q, k_, v_, lens, S, ws, o, cache_batch_idx=idx, k_new=kn,
                               v_new=vn, rope_cos_sin=rope, rope_max_pos=c.cache_len,
                               planned=planned)
        step_outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(step_outs[0].view(torch.int16), step_outs[1].view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))
