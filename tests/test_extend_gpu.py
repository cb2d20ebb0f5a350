"""paged_kv_extend on the GPU against the oracle's extend: the chunk's slots
(V bit for bit, K and the rotated q within one bf16 ulp of the oracle's
single rounding), nothing else touched; and the whole extend step --
paged_kv_extend then paged_prefill_attn -- against the oracle doing the same."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import bits, compare_out, ulp_diff
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _case(lens, qls, ps, Hq, Hkv, D, seed):
    c = wl.prefill("ext", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, page_size=ps, seq_lens=lens,
                   q_lens=qls, seed=seed)
    g = torch.Generator().manual_seed(seed + 11)
    total = int(c.qo_indptr[-1])
    k_new = torch.randn(total, Hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(total, Hkv, D, generator=g).to(torch.bfloat16)
    return c, k_new, v_new


def _run(c, k_new, v_new, rope_q=True):
    w = c.w
    t = w.to_device("cuda")
    P = t["k_pool"].shape[0]
    # the chunk's slots start as NaN on the device too
    d = pkv.dims(w.B, w.Hq, w.Hkv, w.D, w.page_size, P, int(w.kv_indices.numel()),
                 w.max_seq_len, w.scale)
    rope = torch.empty(w.max_seq_len, w.D // 2, 2, dtype=torch.float32, device="cuda")
    pkv.rope_table(rope, w.max_seq_len, w.D, 10000.0)
    q = c.q.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_extend(d, q, k_new.cuda(), v_new.cuda(), c.qo_indptr.cuda(), t["k_pool"],
                        t["v_pool"], t["kv_indices"], t["kv_indptr"], t["seq_lens"],
                        rope_cos_sin=rope, rope_max_pos=w.max_seq_len, rope_q=rope_q, status=st)
    torch.cuda.synchronize()
    return d, t, q, int(st.item()) & 0xFFFFFFFF


@pytest.mark.parametrize("ps,Hq,Hkv,D", [(16, 32, 8, 128), (5, 8, 2, 64), (1, 12, 4, 64)])
def test_extend_matches_oracle(ps, Hq, Hkv, D):
    lens, qls = [40, 1, 130, 77, 0, 16], [40, 1, 30, 3, 0, 16]
    c, k_new, v_new = _case(lens, qls, ps, Hq, Hkv, D, seed=ps + D)
    w = c.w
    t0 = w.to_device("cuda")
    kp0, vp0 = bits(t0["k_pool"]).copy(), bits(t0["v_pool"]).copy()
    del t0
    d, t, q, st = _run(c, k_new, v_new)
    assert st == 0
    q2, kp2, vp2 = oracle.extend(bits(c.q), bits(k_new), bits(v_new), c.qo_indptr.numpy(), kp0,
                                 vp0, w.host("kv_indices"), w.host("kv_indptr"),
                                 w.host("seq_lens"), rope_base=10000.0, rope_q=True)
    assert np.array_equal(bits(t["v_pool"]), vp2)                     # V bit for bit
    kb = bits(t["k_pool"])
    nan = (kp2 & 0x7FFF) > 0x7F80
    assert np.array_equal((kb & 0x7FFF) > 0x7F80, nan)
    assert ulp_diff(kb[~nan], kp2[~nan]).max() <= 1                  # K rotated in fp32
    assert ulp_diff(bits(q), q2).max() <= 1                           # q rotated in place


def test_extend_then_prefill_is_the_extend_step():
    lens, qls = [300, 90, 33, 1], [120, 90, 1, 1]
    c, k_new, v_new = _case(lens, qls, 16, 32, 8, 128, seed=9)
    w = c.w
    t0 = w.to_device("cuda")
    kp0, vp0 = bits(t0["k_pool"]).copy(), bits(t0["v_pool"]).copy()
    del t0
    d, t, q, st = _run(c, k_new, v_new)
    out = torch.empty(c.total_q, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_prefill_attn(d, q, c.qo_indptr.cuda(), t["k_pool"], t["v_pool"], t["kv_indices"],
                           t["kv_indptr"], t["seq_lens"], out, status=st2, max_q_len=max(qls))
    torch.cuda.synchronize()
    assert st == 0 and int(st2.item()) == 0
    q2, kp2, vp2 = oracle.extend(bits(c.q), bits(k_new), bits(v_new), c.qo_indptr.numpy(), kp0,
                                 vp0, w.host("kv_indices"), w.host("kv_indptr"),
                                 w.host("seq_lens"), rope_base=10000.0, rope_q=True)
    want = oracle.prefill(q2, c.qo_indptr.numpy(), kp2, vp2, w.host("kv_indices"),
                          w.host("kv_indptr"), w.host("seq_lens"), w.scale)
    compare_out(out, want)


def test_extend_flags_bad_chunk():
    lens, qls = [50, 20], [10, 20]
    c, k_new, v_new = _case(lens, qls, 16, 8, 2, 64, seed=2)
    c.w.seq_lens[1] = 10                       # row 1's chunk of 20 now exceeds its length
    d, t, q, st = _run(c, k_new, v_new, rope_q=False)
    assert st & pkv.FLAG_BAD_LEN
