"""Kernels (2) and (3), split-KV paged GQA decode + combine, against the
fp64 oracle on the GPU, through the C ABI.

The pools carry NaN in every unreferenced page and in every slot past a
row's end, so a stray read shows up as a non-finite output.  Tolerance
(bf16 output vs fp64): max-abs 2e-2, mean-abs 2e-3."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import GpuCase, bf16_to_f64, bf16_ulp, compare_out, oracle_step
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _full_step(w, num_splits=None, **kw):
    ref = oracle_step(w)
    c = GpuCase(w, num_splits=num_splits, **kw)
    c.append()
    out = c.decode()
    errs = compare_out(out, ref["out"])
    assert c.status() == 0
    return c, ref, errs


# ---- the five workloads, in the launch configuration the benchmark uses ---
@pytest.mark.parametrize("name", ["tiny", "gqa_1b", "ragged_b32", "long_32k"])
def test_workloads_planned(name):
    _full_step(wl.make(name))


@pytest.mark.parametrize("B", wl.SERVING_BATCHES)
def test_serving_mix_planned(B):
    c, ref, _ = _full_step(wl.serving(B))
    # padded rows (seq_len 0) are exactly zero
    pad = (c.w.seq_lens == 0).numpy()
    if pad.any():
        assert torch.count_nonzero(c.out[torch.from_numpy(pad).cuda()]) == 0


# Split invariance, element by element.  Splitting a row changes only the
# rounding: each piece exponentiates against its own running max, so the
# probabilities P, rounded to bf16 before P.V, round differently; the fp32
# merge then rescales them exactly up to fp32 rounding.  A relative change of
# at most 2^-8 in each weight moves an output by 2^-8 * sum_i p_i |v_i - o| at
# most, which for a long row's many small, independently rounded weights
# averages out to far below that; the two bf16 results are each rounded once
# (half an ulp apiece).  The bound is therefore 2 ulp of the larger of the
# two values plus an absolute floor of 2^-10 for outputs near zero, where the
# ulp vanishes but the weights' rounding does not.  It is tighter than the
# oracle tolerance (2e-2) each split already meets, so an error that depends
# on the split (a dropped piece, a wrong rescale) fails it.
SPLIT_ULPS = 2
SPLIT_FLOOR = 2.0 ** -10


def assert_split_invariant(a: torch.Tensor, b: torch.Tensor, what):
    x, y = bf16_to_f64(a), bf16_to_f64(b)
    bound = SPLIT_ULPS * bf16_ulp(np.maximum(np.abs(x), np.abs(y))) + SPLIT_FLOOR
    diff = np.abs(x - y)
    bad = diff > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements differ beyond the bound, "
                           f"worst {diff.max():.3e}")


def test_long_context_split_sweep():
    """Long-context row, every split count 1..256: all within tolerance, and
    S = 1 (one block, no combine) agrees with every other S element by
    element within the split-invariance bound."""
    w = wl.long_32k()
    ref = oracle_step(w)
    c = GpuCase(w, num_splits=256)
    c.append()
    outs = {}
    for S in (1, 2, 4, 8, 16, 32, 64, 128, 256, pkv.plan(c.d)[0]):
        outs[S] = c.decode(S).clone()
        compare_out(outs[S], ref["out"])
    for S, o in outs.items():
        assert_split_invariant(o, outs[1], f"S={S} vs S=1")


@pytest.mark.parametrize("name", ["gqa_1b", "ragged_b32"])
def test_split_invariance_batched(name):
    """Many rows: the planned split (rows cut across blocks, merged by the
    combine) against one split per row (every row whole in one block)."""
    w = wl.make(name)
    c = GpuCase(w)
    c.append()
    planned = c.decode().clone()
    one = c.decode(1).clone()
    assert_split_invariant(planned, one, f"{name}: S={c.S} vs S=1")


# ---- shapes: page sizes, GQA ratios, head dims, ragged tails ------------
@pytest.mark.parametrize("ps", [1, 2, 5, 8, 16, 32, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_page_sizes(ps, D):
    lens = [1, 15, 16, 17, 100, 257, 0, 513]
    w = wl.build("ps", B=len(lens), Hq=16, Hkv=4, D=D, page_size=ps, seq_lens=lens,
                 seed=ps * 7 + D)
    for S in (1, 3):
        _full_step(w, num_splits=S)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (16, 4), (32, 4), (64, 4), (48, 3), (12, 4)])
def test_gqa_ratios(Hq, Hkv):
    lens = [33, 300, 1, 64]
    w = wl.build("gqa", B=4, Hq=Hq, Hkv=Hkv, D=128, page_size=16, seq_lens=lens,
                 seed=Hq + 100 * Hkv)
    _full_step(w, num_splits=2)


def test_capacity_above_lengths():
    # the split grid is sized for a capacity far above the live lengths
    w = wl.build("cap", B=3, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=[40, 1000, 7],
                 seed=8, max_seq_len=8192)
    for S in (1, 4, 32):
        _full_step(w, num_splits=S)


@pytest.mark.parametrize("S", [1, 4])
def test_many_rows_fallback_path(S):
    # more than 4096 virtual rows (Hkv = 1): the per-(split, head, row) kernel
    # and the standalone combine serve the call
    g = torch.Generator().manual_seed(3)
    lens = torch.randint(0, 40, (4200,), generator=g).tolist()
    w = wl.build("many", B=4200, Hq=2, Hkv=1, D=64, page_size=16, seq_lens=lens, seed=3)
    _full_step(w, num_splits=S)


def test_all_rows_empty():
    w = wl.build("empty", B=3, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[0, 0, 0], seed=1,
                 max_seq_len=64)
    for S in (1, 4):
        c = GpuCase(w, num_splits=S)
        c.out.fill_(1.0)
        out = c.decode()
        assert torch.count_nonzero(out) == 0


# ---- the split kernel's partials and the combine on their own ----------
@pytest.mark.parametrize("S", [1, 3, 8])
def test_partials_match_oracle(S):
    w = wl.build("parts", B=4, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[1, 200, 700, 0],
                 seed=31, max_seq_len=800, fill_new_slot=True)
    c = GpuCase(w, num_splits=S)
    t = c.t
    pkv.paged_decode_partials(c.d, t["q"], t["k_pool"], t["v_pool"], t["kv_indices"],
                              t["kv_indptr"], t["seq_lens"], S, c.ws)
    o_gpu, ml_gpu = pkv.partial_views(c.d, S, c.ws)
    o_gpu = o_gpu.cpu().numpy().astype(np.float64)
    ml_gpu = ml_gpu.cpu().numpy().astype(np.float64)
    kp, vp, idx = w.compact_host()
    chunk = pkv.split_chunk(c.d, S)
    o_ref, ml_ref = oracle.decode_partials(w.host("q"), kp, vp, idx, w.host("kv_indptr"),
                                           w.host("seq_lens"), w.scale, S, chunk)
    empty = ml_ref[..., 1] == 0
    assert np.array_equal(empty, ml_gpu[..., 1] == 0)
    assert np.all(ml_gpu[..., 0][empty] == -np.inf)
    full = ~empty
    np.testing.assert_allclose(ml_gpu[..., 0][full], ml_ref[..., 0][full], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(ml_gpu[..., 1][full], ml_ref[..., 1][full], rtol=4e-3)
    err = np.abs(o_gpu[full] - o_ref[full])
    assert err.max() < 1e-2 and err.mean() < 1e-3


def test_combine_matches_oracle():
    g = torch.Generator().manual_seed(5)
    B, Hq, S, D = 3, 8, 37, 128
    o = torch.randn(B, Hq, S, D, generator=g)
    m = torch.randn(B, Hq, S, generator=g) * 4
    l = torch.rand(B, Hq, S, generator=g) * 50 + 0.5
    empty = torch.rand(B, Hq, S, generator=g) < 0.3
    m[empty] = float("-inf")
    l[empty] = 0.0
    o[empty] = float("nan")          # never read for empty splits
    empty_all = torch.zeros(B, Hq, S, dtype=torch.bool)
    empty_all[1, 3] = True           # one (row, head) with every split empty
    m[empty_all] = float("-inf")
    l[empty_all] = 0.0
    ml = torch.stack([m, l], dim=-1).contiguous()
    want = oracle.combine(o.numpy(), ml.numpy())
    d = pkv.dims(B, Hq, 2, D, 16, 1, 0, 16 * S)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    pkv.decode_combine(d, o.cuda(), ml.cuda(), S, out)
    got = bf16_to_f64(out)
    assert np.all(got[1, 3] == 0.0)
    np.testing.assert_allclose(got, np.nan_to_num(want), rtol=2.0 ** -8, atol=1e-6)


def test_repeatable_bitwise():
    w = wl.make("gqa_1b")
    c = GpuCase(w)
    c.append()
    a = c.decode().clone()
    b = c.decode().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
