"""Kernel (1), fused RoPE + K/V append, against the oracle on the GPU.

Indexing is checked bit-exactly over the whole pool: after the append,
exactly the B * Hkv * D elements of each pool at the new tokens' slots have
changed, V there equals v_new bit for bit, and every other element (NaN
sentinels included) is untouched.  Rotated K and q are within one bf16 ulp
of the oracle's single rounding of the fp64 rotation."""

import numpy as np
import pytest
import torch

from gpu_cases import GpuCase, bits, oracle_step, ulp_diff
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _check_append(w, rope_q=True):
    ref = oracle_step(w, rope_q=rope_q)
    c = GpuCase(w)
    k_before = bits(c.t["k_pool"])
    v_before = bits(c.t["v_pool"])
    c.append(rope_q=rope_q)
    assert c.status() == 0
    k_after = bits(c.t["k_pool"])
    v_after = bits(c.t["v_pool"])
    live = int((w.seq_lens > 0).sum())
    n_new = live * w.Hkv * w.D
    assert int((v_after != v_before).sum()) == n_new
    assert int((k_after != k_before).sum()) == n_new
    # referenced pages: V bit-exact, K within 1 ulp of the oracle
    idx = w.kv_indices.numpy().astype(np.int64)
    assert np.array_equal(v_after[idx], ref["v_pages"])
    du = ulp_diff(k_after[idx], ref["k_pages"])
    assert du.max() <= 1, f"K off by {du.max()} ulp"
    # q rotated in place (or untouched)
    dq = ulp_diff(bits(c.t["q"]), ref["q"])
    assert dq.max() <= 1
    return float((du > 0).mean()), float((dq > 0).mean())


@pytest.mark.parametrize("name", ["tiny", "gqa_1b", "serving_b8"])
def test_append_matches_oracle(name):
    frac_k, frac_q = _check_append(wl.make(name))
    # a 1-ulp difference happens only near a rounding tie
    assert frac_k < 0.01 and frac_q < 0.01


@pytest.mark.parametrize("ps", [1, 3, 8, 16, 64])
def test_append_page_sizes(ps):
    w = wl.build("ps", B=5, Hq=8, Hkv=2, D=64, page_size=ps, seq_lens=[1, 2, 17, 64, 130],
                 seed=ps)
    _check_append(w)


def test_append_position_zero_and_padding_rows():
    # seq_len 1 -> position 0: K equals k_new bit for bit; seq_len 0 rows untouched
    w = wl.build("p0", B=4, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[1, 0, 33, 0], seed=3)
    _check_append(w)
    c = GpuCase(w)
    c.append()
    page = int(w.kv_indices[int(w.kv_indptr[0])])
    assert np.array_equal(bits(c.t["k_pool"][page, 0]), bits(w.k_new[0]))


def test_append_without_rope():
    w = wl.build("norope", B=3, Hq=4, Hkv=2, D=64, page_size=16, seq_lens=[5, 16, 40],
                 seed=4, rope_base=None)
    ref = oracle_step(w, rope_q=False)
    c = GpuCase(w)
    c.append(rope_q=False)
    idx = w.kv_indices.numpy().astype(np.int64)
    assert np.array_equal(bits(c.t["k_pool"])[idx], ref["k_pages"])


def test_rope_table_close_to_fp64():
    D, P = 128, 40000
    t = torch.empty(P, D // 2, 2, dtype=torch.float32, device="cuda")
    pkv.rope_table(t, P, D, 10000.0)
    torch.cuda.synchronize()
    pos = np.arange(P, dtype=np.float64)[:, None]
    theta = 10000.0 ** (-2.0 * np.arange(D // 2) / D)
    ang = pos * theta
    got = t.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got[..., 0] - np.cos(ang))) < 1e-7
    assert np.max(np.abs(got[..., 1] - np.sin(ang))) < 1e-7
