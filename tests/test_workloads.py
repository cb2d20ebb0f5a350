"""Seeded workload generator: determinism, shapes and the layout facts the
library relies on (CPU only)."""

import numpy as np
import pytest
import torch

from paged_kv_gqa_16_gb300 import workloads as wl


def test_deterministic():
    a, b = wl.gqa_1b(seed=0), wl.gqa_1b(seed=0)
    for name in ("seq_lens", "kv_indptr", "kv_indices"):
        assert torch.equal(getattr(a, name), getattr(b, name))
    for name in ("q", "k_new", "v_new", "k_pages", "v_pages"):
        assert torch.equal(getattr(a, name).view(torch.int16), getattr(b, name).view(torch.int16))
    c = wl.gqa_1b(seed=1)
    assert not torch.equal(a.seq_lens, c.seq_lens)


@pytest.mark.parametrize("name", ["tiny", "gqa_1b", "long_32k", "serving_b1", "serving_b8",
                                  "serving_b128"])
def test_layout_facts(name):
    w = wl.make(name)
    lens = w.seq_lens.numpy()
    ptr = w.kv_indptr.numpy()
    idx = w.kv_indices.numpy()
    assert ptr[0] == 0 and len(ptr) == w.B + 1
    np.testing.assert_array_equal(np.diff(ptr), -(-lens // w.page_size))
    assert len(np.unique(idx)) == len(idx)                 # distinct pages
    assert idx.min() >= 0 and idx.max() < w.num_pages
    assert lens.max() <= w.max_seq_len
    assert w.q.shape == (w.B, w.Hq, w.D) and w.k_new.shape == (w.B, w.Hkv, w.D)
    # NaN exactly from the new-token slot to the end of each row's last page
    kp = w.k_pages.float()
    for b, L in enumerate(lens):
        if L == 0:
            continue
        rows = kp[ptr[b]:ptr[b + 1]].reshape(-1, w.Hkv, w.D)
        assert torch.isfinite(rows[:L - 1]).all()
        assert torch.isnan(rows[L - 1:]).all()


def test_case_parameters():
    t = wl.tiny()
    assert t.seq_lens.tolist() == [37, 100] and t.num_pages == 16
    g = wl.gqa_1b()
    assert (g.B, g.Hq, g.Hkv, g.D) == (8, 32, 8, 64)
    assert all(513 <= x <= 1025 for x in g.seq_lens.tolist())
    lc = wl.long_32k()
    assert lc.seq_lens.tolist() == [32768] and lc.num_pages == 4096
    s = wl.serving(128)
    lens = s.seq_lens.numpy()
    assert (lens > 0).sum() == 96 and np.all(lens[96:] == 0)
    assert lens[:96].min() >= 16 and lens[:96].max() <= 8192
    assert abs(np.median(np.log(lens[:96])) - np.log(1024)) < 0.5


@pytest.mark.slow
def test_ragged_b32_shape():
    w = wl.ragged_b32()
    lens = w.seq_lens.numpy()
    assert w.B == 32 and w.D == 128 and w.num_pages == 65536
    assert lens.min() >= 512 and lens.max() <= 4096
