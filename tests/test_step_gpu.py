"""paged_decode_step -- append + split decode + combine in one pass -- on the
GPU: bit-identical to paged_kv_append (on a copy of q) followed by
paged_decode_attn, the same pool afterwards, q left unchanged, and within
tolerance of the oracle."""

import numpy as np
import pytest
import torch

from gpu_cases import GpuCase, bits, compare_out, oracle_step
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _step(c, S=None):
    t = c.t
    pkv.paged_decode_step(c.d, t["q"], t["k_new"], t["v_new"], t["k_pool"], t["v_pool"],
                          t["kv_indices"], t["kv_indptr"], t["seq_lens"],
                          c.rope if c.w.rope_base else None, c.rope_max_pos,
                          c.S if S is None else S, c.ws, c.out)
    return c.out


def _check(w, S=None):
    ref = oracle_step(w)
    a = GpuCase(w, num_splits=S)            # fused step
    b = GpuCase(w, num_splits=S)            # separate append + decode
    q_before = bits(a.t["q"])
    out_a = _step(a).clone()
    b.append(rope_q=True)
    out_b = b.decode().clone()
    assert a.status() == 0 and b.status() == 0
    assert np.array_equal(bits(a.t["q"]), q_before)                 # q untouched
    assert np.array_equal(bits(a.t["k_pool"]), bits(b.t["k_pool"]))
    assert np.array_equal(bits(a.t["v_pool"]), bits(b.t["v_pool"]))
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    compare_out(out_a, ref["out"])


@pytest.mark.parametrize("name", ["tiny", "gqa_1b", "ragged_b32", "long_32k", "serving_b1",
                                  "serving_b32", "serving_b128"])
def test_step_planned(name):
    _check(wl.make(name))


@pytest.mark.parametrize("S", [1, 2, 7, 64])
@pytest.mark.parametrize("ps", [1, 5, 16, 32])
def test_step_splits_and_pages(S, ps):
    lens = [1, 2, 15, 16, 17, 31, 100, 0, 301]
    w = wl.build("stp", B=len(lens), Hq=16, Hkv=4, D=128, page_size=ps, seq_lens=lens,
                 seed=S * 10 + ps)
    _check(w, S)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (48, 3, 128), (12, 4, 64), (64, 8, 128)])
def test_step_head_shapes(Hq, Hkv, D):
    w = wl.build("sth", B=3, Hq=Hq, Hkv=Hkv, D=D, page_size=16, seq_lens=[5, 77, 200], seed=Hq)
    _check(w, 3)


def test_step_without_rope():
    w = wl.build("stn", B=3, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[5, 20, 40], seed=2,
                 rope_base=None)
    ref = oracle_step(w, rope_q=False)
    a = GpuCase(w, num_splits=2)
    compare_out(_step(a), ref["out"])


@pytest.mark.parametrize("S", [1, 4])
def test_step_fallback_path(S):
    # > 4096 virtual rows: rotated q copy in the workspace + append + split decode
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(0, 40, (4200,), generator=g).tolist()
    w = wl.build("stf", B=4200, Hq=2, Hkv=1, D=64, page_size=16, seq_lens=lens, seed=4)
    _check(w, S)


@pytest.mark.parametrize("seed", [0, 1])
def test_step_many_short_rows(seed):
    """Hundreds of rows of 0-40 tokens.  Every block's range holds several
    rows' fixed partition weight, some ranges end inside a row's weight
    before its first token, and most rows are single pieces."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, 41, (600,), generator=g)
    lens[::7] = 0
    lens[1::11] = 1
    w = wl.build("short", B=600, Hq=8, Hkv=8, D=64, page_size=16, seq_lens=lens.tolist(),
                 seed=seed)
    _check(w)
    _check(w, 152)
