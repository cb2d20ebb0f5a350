"""paged_decode_attn_noalloc: the decode for callers that cannot allocate
device memory (an allocator-owning runtime, an execute phase that forbids
cudaMalloc), whose workspace is a fixed array held by the library.  Its
output must match paged_decode_attn with a caller workspace, on two calls in
a row with different inputs (the shared array keeps the previous call's
contents, which must not leak into the next).  This file is collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

from gpu_cases import GpuCase, MAX_ABS, MEAN_ABS, bf16_to_f64, compare_out, oracle_step
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(c, status):
    t = c.t
    out = torch.empty_like(c.out)
    out.fill_(float("nan"))
    code = pkv.lib().paged_decode_attn_noalloc(
        ctypes.byref(c.d), t["q"].data_ptr(), t["k_pool"].data_ptr(), t["v_pool"].data_ptr(),
        t["kv_indices"].data_ptr(), t["kv_indptr"].data_ptr(), t["seq_lens"].data_ptr(),
        c.S, out.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == pkv.PKV_OK, pkv.status_str(code)
    return out


def test_noalloc_matches_workspace_call_twice():
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # two calls in a row, same shape, different lengths, tables and values
    for w in (wl.gqa_1b(seed=0), wl.gqa_1b(seed=1)):
        c = GpuCase(w)
        assert pkv.workspace_bytes(c.d, c.S) <= pkv.NOALLOC_SCRATCH_BYTES
        c.append()
        want = c.decode().clone()
        got = _noalloc(c, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        g, r = bf16_to_f64(got), bf16_to_f64(want)
        assert np.all(np.isfinite(g))
        err = np.abs(g - r)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
        compare_out(got, oracle_step(w)["out"])


def test_noalloc_rejects_oversized_shape():
    # a shape whose workspace exceeds the fixed array is refused up front
    d = pkv.dims(4096, 64, 8, 128, 16, 1 << 20, 1 << 20, 8192)
    assert pkv.workspace_bytes(d, 152) > pkv.NOALLOC_SCRATCH_BYTES
    fake = 1 << 32
    code = pkv.lib().paged_decode_attn_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake,
                                               fake, 152, fake, None, None)
    assert code == pkv.PKV_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_empty_batch_clears_status():
    # B = 0 computes nothing, but the caller's status word still starts the
    # call at zero, as every other call leaves it
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    d = pkv.dims(0, 32, 8, 128, 16, 64, 0, 1024)
    code = pkv.lib().paged_decode_attn_noalloc(ctypes.byref(d), None, None, None, None, None,
                                               None, 4, None, status.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert code == pkv.PKV_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("case,want", [
    ("splits_zero", pkv.PKV_ERR_INVALID_ARG),
    ("splits_above_max", pkv.PKV_ERR_INVALID_ARG),
    ("hq_not_multiple", pkv.PKV_ERR_INVALID_ARG),
    ("bad_head_dim", pkv.PKV_ERR_UNSUPPORTED),
])
def test_noalloc_rejects_like_workspace_call(case, want):
    # bad arguments get the codes paged_decode_attn gives them
    d = pkv.dims(4, 32, 8, 128, 16, 64, 64, 1024)
    S = 4
    if case == "splits_zero":
        S = 0
    elif case == "splits_above_max":
        S = 65537
    elif case == "hq_not_multiple":
        d.Hq = 30
    elif case == "bad_head_dim":
        d.D = 96
    fake = 1 << 32
    ref = pkv.lib().paged_decode_attn(ctypes.byref(d), fake, fake, fake, fake, fake, fake, S,
                                      fake, 1 << 30, fake, None)
    code = pkv.lib().paged_decode_attn_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake,
                                               fake, S, fake, None, None)
    assert code == ref == want

