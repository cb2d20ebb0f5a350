"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not share code with:
hand-derived golden values (tests/golden/, with their derivations), closed
forms of softmax attention, invariants the definition fixes, and special
cases that reduce to library routines (torch's binary32->bf16 rounding,
torch complex multiplication, torch scaled_dot_product_attention in fp64).
"""

import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_gqa_16_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- bf16 ---
def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def test_bf16_rne_golden():
    n = 0
    for row in _golden_rows("bf16_rne.txt"):
        x_hex, bits_hex = row.split()[:2]
        x = float.fromhex(x_hex)
        got = int(oracle.bf16_round(np.array([x]))[0])
        assert got == int(bits_hex, 16), f"{x_hex}: got {got:#06x}, want {bits_hex}"
        n += 1
    assert n >= 15


def test_bf16_rne_matches_torch_on_binary32_values():
    # For inputs already in binary32 there is one rounding only, and torch's
    # float -> bfloat16 conversion is round-to-nearest-even.
    g = torch.Generator().manual_seed(1)
    bits = torch.randint(0, 2**31 - 1, (200000,), generator=g, dtype=torch.int64)
    bits = bits.to(torch.int32)
    f = bits.view(torch.float32)
    f = f[torch.isfinite(f)]
    # plenty of exact ties: low 16 bits = 0x8000
    ties = (torch.randint(0, 2**15, (5000,), generator=g, dtype=torch.int32) << 16) | 0x8000
    f = torch.cat([f, ties.view(torch.float32), -f[:1000]])
    f = f[torch.isfinite(f)]
    want = f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(f.to(torch.float64).numpy())
    assert np.array_equal(got, want)


def test_bf16_widening_is_exact_roundtrip():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = oracle.bf16_to_f64(allbits)
    finite = np.isfinite(x)
    back = oracle.bf16_round(x[finite])
    assert np.array_equal(back, allbits[finite])
    ref = torch.from_numpy(allbits.astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    assert np.array_equal(x[finite], ref.numpy()[finite])


# ----------------------------------------------------------------- RoPE ---
def _eval_expr(s):
    return float(eval(s, {"cos": math.cos, "sin": math.sin, "__builtins__": {}}))


def test_rope_golden():
    n = 0
    for row in _golden_rows("rope_cases.txt"):
        D, base, pos, xs, ys = [c.strip() for c in row.split("|")]
        x = np.array([float(v) for v in xs.split(",")])
        want = np.array([_eval_expr(v) for v in ys.split(",")])
        got = oracle.rope_rotate(x, int(pos), float(base))
        assert x.size == int(D)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
        n += 1
    assert n >= 6


def _torch_complex_rope(x, pos, base):
    # The pages' training path: view pairs as complex numbers, multiply by
    # a unit phasor built with torch.polar.
    D = x.size
    i = torch.arange(D // 2, dtype=torch.float64)
    theta = base ** (-2.0 * i / D)
    rot = torch.polar(torch.ones_like(theta), pos * theta)
    xc = torch.view_as_complex(torch.from_numpy(x.copy()).view(D // 2, 2))
    return torch.view_as_real(xc * rot).reshape(D).numpy()


@pytest.mark.parametrize("D", [8, 64, 128])
@pytest.mark.parametrize("pos", [0, 1, 17, 1023, 32767])
def test_rope_matches_torch_complex_multiply(D, pos):
    x = np.random.default_rng(D + pos).standard_normal(D)
    got = oracle.rope_rotate(x, pos, 10000.0)
    want = _torch_complex_rope(x, pos, 10000.0)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(3)
    D = 64
    q = rng.standard_normal(D)
    k = rng.standard_normal(D)
    # pair norms preserved
    y = oracle.rope_rotate(q, 777, 10000.0)
    np.testing.assert_allclose(np.hypot(y[0::2], y[1::2]), np.hypot(q[0::2], q[1::2]),
                               rtol=1e-14)
    # composition: R_a R_b = R_{a+b}
    y2 = oracle.rope_rotate(oracle.rope_rotate(q, 300, 10000.0), 477, 10000.0)
    np.testing.assert_allclose(y2, y, atol=1e-11)
    # inner product depends only on the position difference
    a = oracle.rope_rotate(q, 50, 10000.0) @ oracle.rope_rotate(k, 20, 10000.0)
    b = oracle.rope_rotate(q, 1030, 10000.0) @ oracle.rope_rotate(k, 1000, 10000.0)
    assert abs(a - b) < 1e-10


# --------------------------------------------------------------- append ---
def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_append_touches_exactly_the_new_slots():
    w = wl.tiny()
    kp, vp = w.full_pool_host()
    q2, kp2, vp2 = oracle.append(w.host("q"), w.host("k_new"), w.host("v_new"), kp, vp,
                                 w.host("kv_indices"), w.host("kv_indptr"),
                                 w.host("seq_lens"), rope_base=10000.0, rope_q=False)
    assert np.array_equal(q2, w.host("q"))
    changed_k = np.argwhere(kp2 != kp)
    changed_v = np.argwhere(vp2 != vp)
    # every element of the new slot was NaN before and is finite after
    assert len(changed_k) == w.B * w.Hkv * w.D
    assert len(changed_v) == w.B * w.Hkv * w.D
    idx = w.kv_indices.numpy()
    ptr = w.kv_indptr.numpy()
    for b in range(w.B):
        pos = int(w.seq_lens[b]) - 1
        page = idx[ptr[b] + pos // w.page_size]
        slot = pos % w.page_size
        # V is copied unchanged
        assert np.array_equal(vp2[page, slot], w.host("v_new")[b])
        # K is the rotated new key, rounded once
        kf = oracle.bf16_to_f64(w.host("k_new")[b])
        for g in range(w.Hkv):
            want = _torch_complex_rope(kf[g], pos, 10000.0)
            got = oracle.bf16_to_f64(kp2[page, slot, g])
            # bf16 spacing near |want| bounds a single rounding
            assert np.all(np.abs(got - want) <= np.abs(want) * 2.0**-8 + 1e-30)


def test_append_position_zero_is_identity_and_rope_q():
    w = wl.build("p0", B=3, Hq=4, Hkv=2, D=16, page_size=4, seq_lens=[1, 5, 9], seed=5)
    kp, vp = w.full_pool_host()
    q2, kp2, vp2 = oracle.append(w.host("q"), w.host("k_new"), w.host("v_new"), kp, vp,
                                 w.host("kv_indices"), w.host("kv_indptr"),
                                 w.host("seq_lens"), rope_base=10000.0, rope_q=True)
    idx, ptr = w.kv_indices.numpy(), w.kv_indptr.numpy()
    # row 0: position 0, cos = 1, sin = 0 -> bit-identical K and q
    assert np.array_equal(kp2[idx[ptr[0]], 0], w.host("k_new")[0])
    assert np.array_equal(q2[0], w.host("q")[0])
    # rows 1, 2: q rotated by the same position as K
    for b in (1, 2):
        pos = int(w.seq_lens[b]) - 1
        qf = oracle.bf16_to_f64(w.host("q")[b])
        for h in range(w.Hq):
            want = _torch_complex_rope(qf[h], pos, 10000.0)
            got = oracle.bf16_to_f64(q2[b, h])
            assert np.all(np.abs(got - want) <= np.abs(want) * 2.0**-8 + 1e-30)


def test_append_without_rope_copies_k():
    w = wl.build("norope", B=2, Hq=2, Hkv=1, D=8, page_size=2, seq_lens=[3, 6], seed=6)
    kp, vp = w.full_pool_host()
    _, kp2, _ = oracle.append(w.host("q"), w.host("k_new"), w.host("v_new"), kp, vp,
                              w.host("kv_indices"), w.host("kv_indptr"), w.host("seq_lens"),
                              rope_base=None, rope_q=False)
    idx, ptr = w.kv_indices.numpy(), w.kv_indptr.numpy()
    for b in range(2):
        pos = int(w.seq_lens[b]) - 1
        assert np.array_equal(kp2[idx[ptr[b] + pos // 2], pos % 2], w.host("k_new")[b])


# --------------------------------------------------------------- decode ---
def _torch_gather_sdpa(q_bits, kp_bits, vp_bits, kv_indices, kv_indptr, seq_lens, scale):
    """Independent route: torch indexing gathers each row's pages, then
    torch SDPA (fp64, enable_gqa) computes the attention."""
    to64 = lambda a: torch.from_numpy(a.astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    q, kp, vp = to64(q_bits), to64(kp_bits), to64(vp_bits)
    B, Hq, D = q.shape
    P, ps, Hkv, _ = kp.shape
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        pages = torch.from_numpy(kv_indices[kv_indptr[b]:kv_indptr[b + 1]].astype(np.int64))
        K = kp[pages].reshape(-1, Hkv, D)[:L].permute(1, 0, 2)[None]
        V = vp[pages].reshape(-1, Hkv, D)[:L].permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(q[b][None, :, None, :], K, V, scale=scale,
                                           enable_gqa=True)
        out[b] = o[0, :, 0, :]
    return out.numpy()


def _decode_case(w, full=True):
    if full:
        kp, vp = w.full_pool_host()
        idx = w.host("kv_indices")
    else:
        kp, vp, idx = w.compact_host()
    return (w.host("q"), kp, vp, idx, w.host("kv_indptr"), w.host("seq_lens"))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (16, 2), (8, 1), (16, 16)])
@pytest.mark.parametrize("ps", [1, 3, 16, 32])
def test_decode_matches_torch_sdpa(Hq, Hkv, ps):
    lens = [0, 1, 2, 15, 16, 17, 33, 70]
    w = wl.build("sdpa", B=len(lens), Hq=Hq, Hkv=Hkv, D=64, page_size=ps, seq_lens=lens,
                 seed=Hq * 100 + Hkv * 10 + ps, fill_new_slot=True)
    args = _decode_case(w)
    got = oracle.decode(*args, scale=w.scale)
    want = _torch_gather_sdpa(*args, scale=w.scale)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    assert np.all(got[0] == 0.0)            # seq_len 0 row -> zeros


def test_decode_tiny_after_append_is_finite_and_matches_sdpa():
    w = wl.tiny()
    kp, vp = w.full_pool_host()
    _, kp2, vp2 = oracle.append(w.host("q"), w.host("k_new"), w.host("v_new"), kp, vp,
                                w.host("kv_indices"), w.host("kv_indptr"),
                                w.host("seq_lens"), rope_base=10000.0, rope_q=False)
    args = (w.host("q"), kp2, vp2, w.host("kv_indices"), w.host("kv_indptr"),
            w.host("seq_lens"))
    got = oracle.decode(*args, scale=w.scale)
    assert np.all(np.isfinite(got))         # NaN tails / unreferenced pages unread
    np.testing.assert_allclose(got, _torch_gather_sdpa(*args, scale=w.scale), atol=1e-12)


def _single_row(K, V, qv, ps=4):
    """Pool holding one row (one kv head) with keys K [L,D] and values V."""
    L, D = K.shape
    n = -(-L // ps)
    kp = np.full((n, ps, 1, D), wl.NAN_BF16_BITS, dtype=np.uint16)
    vp = kp.copy()
    for t in range(L):
        kp[t // ps, t % ps, 0] = oracle.bf16_round(K[t])
        vp[t // ps, t % ps, 0] = oracle.bf16_round(V[t])
    q = oracle.bf16_round(qv)[None, None, :]
    return q, kp, vp, np.arange(n, dtype=np.int32), np.array([0, n], np.int32), \
        np.array([L], np.int32)


def _exact_bf16(x):
    return oracle.bf16_to_f64(oracle.bf16_round(x))


def test_closed_form_single_token_returns_v0():
    rng = np.random.default_rng(0)
    K, V, qv = rng.standard_normal((1, 32)), rng.standard_normal((1, 32)), rng.standard_normal(32)
    out = oracle.decode(*_single_row(K, V, qv), scale=0.3)
    assert np.array_equal(out[0, 0], _exact_bf16(V[0]))


def test_closed_form_identical_keys_give_mean_v():
    rng = np.random.default_rng(1)
    L, D = 37, 16
    K = np.tile(rng.standard_normal(D), (L, 1))
    V = rng.standard_normal((L, D))
    out = oracle.decode(*_single_row(K, V, rng.standard_normal(D)), scale=1.0)
    np.testing.assert_allclose(out[0, 0], _exact_bf16(V).mean(axis=0), atol=1e-14)


def test_closed_form_zero_query_gives_mean_v():
    rng = np.random.default_rng(2)
    L, D = 21, 16
    K, V = rng.standard_normal((L, D)), rng.standard_normal((L, D))
    out = oracle.decode(*_single_row(K, V, np.zeros(D)), scale=1.0)
    np.testing.assert_allclose(out[0, 0], _exact_bf16(V).mean(axis=0), atol=1e-14)


def test_closed_form_dominant_key():
    # one key aligned with a large query: its weight is 1 up to exp(-gap)
    L, D = 10, 8
    K = np.zeros((L, D))
    K[6, 0] = 1.0
    V = np.arange(L * D, dtype=np.float64).reshape(L, D) / 64.0
    qv = np.zeros(D)
    qv[0] = 64.0
    out = oracle.decode(*_single_row(K, V, qv), scale=1.0)   # gap = 64
    want = _exact_bf16(V[6])
    bound = (L - 1) * math.exp(-64.0) * np.abs(_exact_bf16(V)).max() * 2
    assert np.max(np.abs(out[0, 0] - want)) <= bound


def test_two_token_closed_form():
    # scores s0, s1: out = (v0 + e^(s1-s0) v1) / (1 + e^(s1-s0))
    D = 8
    K = np.zeros((2, D))
    K[0, 0], K[1, 1] = 1.0, 1.0
    qv = np.zeros(D)
    qv[0], qv[1] = 0.5, 2.0                      # s = 0.5, 2.0 at scale 1
    V = np.array([[1.0] * D, [-3.0] * D])
    out = oracle.decode(*_single_row(K, V, qv), scale=1.0)
    e = math.exp(1.5)
    np.testing.assert_allclose(out[0, 0], (1.0 - 3.0 * e) / (1.0 + e), atol=1e-15)


def test_gqa_head_mapping():
    # V of kv head g is the constant g+1, so query head h must return
    # h // n_rep + 1 whatever the scores are.
    Hq, Hkv, D, ps = 8, 2, 16, 4
    w = wl.build("map", B=2, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, seq_lens=[5, 11], seed=9,
                 fill_new_slot=True)
    q, kp, vp, idx, ptr, sl = _decode_case(w, full=False)
    vp = vp.copy()
    for g in range(Hkv):
        vp[:, :, g, :] = oracle.bf16_round(np.full(vp[:, :, g, :].shape, g + 1.0))
    out = oracle.decode(q, kp, vp, idx, ptr, sl, scale=w.scale)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h, :], h // (Hq // Hkv) + 1.0, atol=1e-14)


def test_page_permutation_invariance_is_bitwise():
    w = wl.build("perm", B=3, Hq=8, Hkv=2, D=32, page_size=4, seq_lens=[9, 30, 4],
                 seed=11, fill_new_slot=True)
    q, kp, vp, idx, ptr, sl = _decode_case(w, full=False)
    out = oracle.decode(q, kp, vp, idx, ptr, sl, scale=w.scale)
    perm = np.random.default_rng(4).permutation(kp.shape[0])
    inv = np.argsort(perm)
    out2 = oracle.decode(q, kp[perm], vp[perm], inv[idx].astype(np.int32), ptr, sl,
                         scale=w.scale)
    assert np.array_equal(out, out2)


def test_contiguous_equals_paged_bitwise():
    w = wl.build("contig", B=2, Hq=4, Hkv=2, D=32, page_size=8, seq_lens=[40, 17],
                 seed=12, fill_new_slot=True)
    q, kp, vp, idx, ptr, sl = _decode_case(w, full=False)
    out_paged = oracle.decode(q, kp, vp, idx, ptr, sl, scale=w.scale)
    # one page per row, page_size = 40 (the longest row): a contiguous layout
    Lmax = 40
    kc = np.full((2, Lmax, 2, 32), wl.NAN_BF16_BITS, np.uint16)
    vc = kc.copy()
    for b in range(2):
        K, V = oracle.gather(b, 0, kp, vp, idx, ptr, sl)
        for g in range(2):
            K, V = oracle.gather(b, g, kp, vp, idx, ptr, sl)
            kc[b, :sl[b], g] = oracle.bf16_round(K)
            vc[b, :sl[b], g] = oracle.bf16_round(V)
    out_c = oracle.decode(q, kc, vc, np.array([0, 1], np.int32),
                          np.array([0, 1, 2], np.int32), sl, scale=w.scale)
    assert np.array_equal(out_paged, out_c)


def test_decode_rejects_out_of_range_pages():
    w = wl.build("bad", B=1, Hq=2, Hkv=1, D=8, page_size=4, seq_lens=[6], seed=13,
                 fill_new_slot=True)
    q, kp, vp, idx, ptr, sl = _decode_case(w, full=False)
    with pytest.raises(ValueError):
        oracle.decode(q, kp, vp, np.array([0, kp.shape[0]], np.int32), ptr, sl, scale=1.0)
    with pytest.raises(ValueError):   # table shorter than the row
        oracle.decode(q, kp, vp, idx, np.array([0, 1], np.int32), sl, scale=1.0)


# ------------------------------------------------------ split + combine ---
@pytest.mark.parametrize("chunk", [1, 5, 16, 48, 200])
def test_split_then_combine_equals_direct(chunk):
    lens = [0, 1, 16, 47, 100, 161]
    w = wl.build("split", B=len(lens), Hq=8, Hkv=2, D=32, page_size=16, seq_lens=lens,
                 seed=21, fill_new_slot=True)
    args = _decode_case(w, full=False)
    direct = oracle.decode(*args, scale=w.scale)
    S = -(-max(lens) // chunk)
    o, ml = oracle.decode_partials(*args, scale=w.scale, num_splits=S, chunk=chunk)
    merged = oracle.combine(o, ml)
    np.testing.assert_allclose(merged, direct, rtol=0, atol=1e-13)
    # splits past the end of a row are empty
    for b, L in enumerate(lens):
        n_act = -(-L // chunk)
        assert np.all(ml[b, :, n_act:, 0] == -np.inf)
        assert np.all(ml[b, :, n_act:, 1] == 0.0)
        assert np.all(ml[b, :, :n_act, 1] >= 1.0)     # l >= 1: the max term is e^0


def test_single_split_statistics():
    rng = np.random.default_rng(5)
    L, D = 13, 8
    K, V, qv = rng.standard_normal((L, D)), rng.standard_normal((L, D)), rng.standard_normal(D)
    args = _single_row(K, V, qv)
    o, ml = oracle.decode_partials(*args, scale=0.5, num_splits=1, chunk=64)
    s = 0.5 * (_exact_bf16(K) @ _exact_bf16(qv))
    assert ml[0, 0, 0, 0] == pytest.approx(s.max(), abs=1e-14)
    assert ml[0, 0, 0, 1] == pytest.approx(np.exp(s - s.max()).sum(), rel=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], oracle.decode(*args, scale=0.5)[0, 0], atol=1e-15)


def test_combine_rules():
    rng = np.random.default_rng(6)
    B, Hq, S, D = 2, 3, 5, 8
    o = rng.standard_normal((B, Hq, S, D)).astype(np.float32)
    ml = np.stack([rng.standard_normal((B, Hq, S)) * 3,
                   rng.uniform(0.5, 20, (B, Hq, S))], axis=-1).astype(np.float32)
    out = oracle.combine(o, ml)
    # brute force in the plain weighted-average form
    w = ml[..., 1].astype(np.float64) * np.exp(ml[..., 0].astype(np.float64))
    want = (w[..., None] * o).sum(2) / w.sum(2)[..., None]
    np.testing.assert_allclose(out, want, rtol=1e-12)
    # order of splits does not matter
    p = rng.permutation(S)
    np.testing.assert_allclose(oracle.combine(o[:, :, p], ml[:, :, p]), out, rtol=1e-13)
    # an empty split (l = 0, m = -inf, garbage o) contributes nothing
    o2, ml2 = o.copy(), ml.copy()
    o2[:, :, 2] = np.nan
    ml2[:, :, 2] = (-np.inf, 0.0)
    keep = [0, 1, 3, 4]
    np.testing.assert_allclose(oracle.combine(o2, ml2), oracle.combine(o[:, :, keep],
                                                                       ml[:, :, keep]),
                               rtol=1e-13)
    # every split empty -> zeros; one split -> its own output
    ml3 = ml.copy()
    ml3[..., 0], ml3[..., 1] = -np.inf, 0.0
    assert np.all(oracle.combine(o, ml3) == 0.0)
    np.testing.assert_array_equal(oracle.combine(o[:, :, :1], ml[:, :, :1]),
                                  o[:, :, 0].astype(np.float64))


# -------------------------------------------------------------- advance ---
def test_advance_golden():
    """Hand-worked steps (page_size 4, four table entries per row).

    Row lengths 0, 3, 4, 8, 5, 12, 16: row 0 is idle; rows 1 and 4 grow
    inside their last page (positions 3 and 5); rows 2, 3 and 5 start a page
    (positions 4, 8, 12: page index 1, 2, 3) and take the free pages in row
    order; row 6 (position 16, page index 4) has no fifth entry.  With the
    list [100, 101] from head 0, row 5 finds it empty."""
    ptr = np.arange(8, dtype=np.int32) * 4
    ind = np.full(28, -1, np.int32)
    sl, ind2, head, n_len, n_page, n_bad = oracle.advance(
        [0, 3, 4, 8, 5, 12, 16], ptr, ind, [100, 101], 0, page_size=4, max_seq_len=64)
    assert sl.tolist() == [0, 4, 5, 9, 6, 12, 16]
    want = ind.copy()
    want[2 * 4 + 1] = 100
    want[3 * 4 + 2] = 101
    assert ind2.tolist() == want.tolist()
    assert (head, n_len, n_page, n_bad) == (2, 0, 2, 0)
    # a longer list from head 1: row 5 now gets a page (the list's third)
    sl, ind2, head, _, n_page, _ = oracle.advance(
        [0, 3, 4, 8, 5, 12, 16], ptr, ind, [7, 100, 101, 102], 1, page_size=4, max_seq_len=64)
    assert sl.tolist() == [0, 4, 5, 9, 6, 13, 16]
    assert (ind2[9], ind2[14], ind2[23], head, n_page) == (100, 101, 102, 4, 1)
    # the length bound: position max_seq_len - 1 is the last one allowed
    sl, _, _, n_len, _, _ = oracle.advance([7, 8, 9], np.arange(4, dtype=np.int32) * 4,
                                           np.full(12, 5, np.int32), [1], 0, page_size=4,
                                           max_seq_len=8)
    assert sl.tolist() == [8, 8, 9] and n_len == 2


def test_advance_page_count_over_many_steps():
    """After k steps with a large free list, each live row holds
    ceil((L + k) / ps) pages: the pages taken are the difference, all distinct,
    and they come off the list in order."""
    g = torch.Generator().manual_seed(11)
    B, ps, k, cap = 40, 8, 37, 24
    lens = torch.randint(0, 120, (B,), generator=g).tolist()
    lens[3] = 0
    lens[4] = 8
    ptr = np.arange(B + 1, dtype=np.int32) * cap
    ind = np.full(B * cap, -1, np.int32)
    free = np.arange(1000, 1000 + B * cap, dtype=np.int32)[::-1].copy()
    sl, head = np.array(lens, np.int32), 0
    for _ in range(k):
        sl, ind, head, n_len, n_page, n_bad = oracle.advance(sl, ptr, ind, free, head, ps, 10 ** 6)
        assert n_len == n_page == n_bad == 0
    live = np.array(lens) > 0
    assert np.array_equal(sl, np.where(live, np.array(lens) + k, 0))
    taken = sum(-(-(L + k) // ps) - -(-L // ps) for L in lens if L > 0)
    assert head == taken
    got = ind[ind >= 0]
    assert len(got) == taken and len(set(got.tolist())) == taken
    assert set(got.tolist()) == set(free[:taken].tolist())


# -------------------------------------------------------------- prefill ---
def _prefill_args(c, full=True):
    w = c.w
    if full:
        kp, vp = w.full_pool_host()
        idx = w.host("kv_indices")
    else:
        kp, vp, idx = w.compact_host()
    q = c.q.contiguous().view(torch.int16).numpy().view(np.uint16)
    return q, c.qo_indptr.numpy(), kp, vp, idx, w.host("kv_indptr"), w.host("seq_lens")


def _torch_prefill(q_bits, qo_indptr, kp_bits, vp_bits, kv_indices, kv_indptr, seq_lens, scale):
    """Independent route: torch gathers each row's pages; fp64 SDPA with an
    explicit boolean mask, query i of a chunk of n keeping keys <= L - n + i."""
    to64 = lambda a: torch.from_numpy(a.astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    q, kp, vp = to64(q_bits), to64(kp_bits), to64(vp_bits)
    total_q, Hq, D = q.shape
    P, ps, Hkv, _ = kp.shape
    out = torch.zeros(total_q, Hq, D, dtype=torch.float64)
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        a, e = int(qo_indptr[b]), int(qo_indptr[b + 1])
        n = e - a
        if n == 0:
            continue
        pages = torch.from_numpy(kv_indices[kv_indptr[b]:kv_indptr[b + 1]].astype(np.int64))
        K = kp[pages].reshape(-1, Hkv, D)[:L].permute(1, 0, 2)[None]
        V = vp[pages].reshape(-1, Hkv, D)[:L].permute(1, 0, 2)[None]
        keep = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        o = F.scaled_dot_product_attention(q[a:e].permute(1, 0, 2)[None], K, V,
                                           attn_mask=keep, scale=scale, enable_gqa=True)
        out[a:e] = o[0].permute(1, 0, 2)
    return out.numpy()


@pytest.mark.parametrize("Hq,Hkv,ps", [(8, 2, 16), (4, 4, 1), (16, 2, 5), (8, 1, 32)])
def test_prefill_matches_torch_sdpa(Hq, Hkv, ps):
    lens = [40, 1, 70, 33, 0, 17]
    qls = [40, 1, 9, 33, 0, 1]          # full prefills, extends, single tokens, an idle row
    c = wl.prefill("pf", B=len(lens), Hq=Hq, Hkv=Hkv, D=64, page_size=ps, seq_lens=lens,
                   q_lens=qls, seed=Hq + ps)
    args = _prefill_args(c)
    got = oracle.prefill(*args, scale=c.w.scale)
    want = _torch_prefill(*args, scale=c.w.scale)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_prefill_special_cases():
    lens, qls = [12, 20, 9], [12, 1, 4]
    c = wl.prefill("pfs", B=3, Hq=4, Hkv=2, D=64, page_size=4, seq_lens=lens, q_lens=qls,
                   seed=9)
    args = _prefill_args(c)
    got = oracle.prefill(*args, scale=c.w.scale)
    q, qo, kp, vp, idx, ptr, sl = args
    # a full prefill's first query sees only key 0: its output is V_0 exactly
    for h in range(4):
        v0 = oracle.bf16_to_f64(vp[idx[ptr[0]], 0, h // 2])
        assert np.array_equal(got[0, h], v0)
    # a one-query chunk is the decode of that row
    dec = oracle.decode(q[12:13].reshape(1, 4, 64), kp, vp, idx[ptr[1]:ptr[2]],
                        np.array([0, ptr[2] - ptr[1]], np.int32), np.array([20], np.int32),
                        c.w.scale)
    np.testing.assert_allclose(got[12], dec[0], rtol=0, atol=1e-13)
    # causality: changing the K/V of row 2's last token moves only its last query
    kp2, vp2 = kp.copy(), vp.copy()
    page, slot = idx[ptr[2] + 8 // 4], 8 % 4
    kp2[page, slot] ^= 0x0040
    vp2[page, slot] ^= 0x0040
    got2 = oracle.prefill(q, qo, kp2, vp2, idx, ptr, sl, scale=c.w.scale)
    assert np.array_equal(got2[:16], got[:16])
    assert not np.array_equal(got2[16], got[16])
    # a chunk longer than its row is refused
    with pytest.raises(ValueError):
        oracle.prefill(q, np.array([0, 13, 14, 18], np.int32), kp, vp, idx, ptr, sl,
                       scale=c.w.scale)


# --------------------------------------------------------------- extend ---
def _extend_case(lens, qls, ps, seed, Hq=4, Hkv=2, D=16):
    """Pools with NaN in every chunk slot (the tokens about to be written),
    chunk K/V and q drawn separately."""
    c = wl.prefill("ext", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, page_size=ps, seq_lens=lens,
                   q_lens=qls, seed=seed)
    kp, vp = c.w.full_pool_host()
    idx, ptr = c.w.host("kv_indices"), c.w.host("kv_indptr")
    slots = []
    for b, (L, n) in enumerate(zip(lens, qls)):
        for i in range(n):
            pos = L - n + i
            slots.append((idx[ptr[b] + pos // ps], pos % ps, pos))
    for page, slot, _ in slots:
        kp[page, slot] = wl.NAN_BF16_BITS
        vp[page, slot] = wl.NAN_BF16_BITS
    g = torch.Generator().manual_seed(seed + 1)
    total = int(c.qo_indptr[-1])
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    k_new = bits(torch.randn(total, Hkv, D, generator=g).to(torch.bfloat16))
    v_new = bits(torch.randn(total, Hkv, D, generator=g).to(torch.bfloat16))
    q = bits(c.q)
    return c, q, k_new, v_new, kp, vp, idx, ptr, slots


def test_extend_writes_exactly_the_chunk_slots():
    lens, qls, ps = [6, 3, 9, 0], [3, 3, 1, 0], 4
    c, q, kn, vn, kp, vp, idx, ptr, slots = _extend_case(lens, qls, ps, seed=3)
    q2, kp2, vp2 = oracle.extend(q, kn, vn, c.qo_indptr.numpy(), kp, vp, idx, ptr,
                                 c.w.host("seq_lens"), rope_base=10000.0, rope_q=False)
    assert np.array_equal(q2, q)
    assert len(np.argwhere(kp2 != kp)) == len(slots) * 2 * 16     # NaN -> finite, all of it
    assert len(np.argwhere(vp2 != vp)) == len(slots) * 2 * 16
    for t, (page, slot, pos) in enumerate(slots):
        assert np.array_equal(vp2[page, slot], vn[t])              # V copied
        kf = oracle.bf16_to_f64(kn[t])
        for gg in range(2):
            want = _torch_complex_rope(kf[gg], pos, 10000.0)
            got = oracle.bf16_to_f64(kp2[page, slot, gg])
            assert np.all(np.abs(got - want) <= np.abs(want) * 2.0**-8 + 1e-30)
        if pos == 0:
            assert np.array_equal(kp2[page, slot], kn[t])          # angle 0: identity


def test_extend_one_token_is_append_and_rotates_q():
    lens, ps = [5, 1, 12], 4
    c, q, kn, vn, kp, vp, idx, ptr, slots = _extend_case(lens, [1, 1, 1], ps, seed=4)
    e = oracle.extend(q, kn, vn, c.qo_indptr.numpy(), kp, vp, idx, ptr, c.w.host("seq_lens"),
                      rope_base=10000.0, rope_q=True)
    a = oracle.append(q, kn, vn, kp, vp, idx, ptr, c.w.host("seq_lens"), rope_base=10000.0,
                      rope_q=True)
    for x, y in zip(e, a):
        assert np.array_equal(x, y)
    # the chunk's query heads are rotated by their token's position
    qf = oracle.bf16_to_f64(q)
    for t, (_, _, pos) in enumerate(slots):
        for h in range(4):
            want = _torch_complex_rope(qf[t, h], pos, 10000.0)
            got = oracle.bf16_to_f64(e[0][t, h])
            assert np.all(np.abs(got - want) <= np.abs(want) * 2.0**-8 + 1e-30)
    with pytest.raises(ValueError):                                 # chunk longer than its row
        oracle.extend(q, kn, vn, np.array([0, 1, 3, 3], np.int32), kp, vp, idx, ptr,
                      c.w.host("seq_lens"), rope_base=None, rope_q=False)
