"""Device-side checks: invalid tables and lengths are turned into status
flags by the kernels' own bounds checks (an out-of-range page is replaced
by page 0, never dereferenced), so the GPU never faults and the context
stays usable.  These run only after the parity tests have passed."""

import pytest
import torch

from gpu_cases import GpuCase, compare_out, oracle_step
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _case(**kw):
    w = wl.build("err", B=3, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[20, 40, 5], seed=2,
                 **kw)
    return w, GpuCase(w, num_splits=2)


@pytest.mark.parametrize("bad_page", [-1, 10**6])
def test_out_of_range_page_sets_flag(bad_page):
    w, c = _case()
    c.t["kv_indices"][1] = bad_page
    c.decode()
    assert c.status() & pkv.FLAG_BAD_PAGE
    pkv.workspace_init(c.ws)
    c.append()
    assert c.status() & pkv.FLAG_BAD_PAGE


def test_length_above_capacity_sets_flag():
    w, c = _case()
    c.t["seq_lens"][0] = w.max_seq_len + 1
    c.decode()
    assert c.status() & pkv.FLAG_BAD_LEN


def test_short_table_sets_flag():
    w, c = _case()
    c.t["kv_indptr"][1] = c.t["kv_indptr"][0]      # row 0 has no pages
    c.decode()
    assert c.status() & pkv.FLAG_BAD_PAGE


def test_rope_position_past_table_sets_flag():
    w, c = _case()
    c.rope_max_pos = 10                             # rows of length 20, 40 are past it
    c.append()
    assert c.status() & pkv.FLAG_BAD_POS


def test_context_usable_after_flags():
    w, c = _case()
    c.t["kv_indices"][0] = 10**6
    c.decode()
    assert c.status() & pkv.FLAG_BAD_PAGE
    # a clean case still computes correctly afterwards
    w2 = wl.make("tiny")
    c2 = GpuCase(w2)
    c2.append()
    compare_out(c2.decode(), oracle_step(w2)["out"])
    assert c2.status() == 0


def test_handoff_timeout_sets_flag_and_context_survives():
    """The bounded waits' own path: with the hand-off limit at zero, the
    decode kernel's producer and consumer warps give up waiting on each other
    while copies are in flight.  The call still returns, the status word
    carries PKV_FLAG_TIMEOUT, and once the limit is back a normal call on the
    same context matches the oracle."""
    w = wl.make("gqa_1b")
    c = GpuCase(w)
    c.append()
    try:
        pkv.testing_set_handoff_wait_ns(0)
        for _ in range(3):
            pkv.workspace_init(c.ws)
            c.decode()
            assert c.status() & pkv.FLAG_TIMEOUT
    finally:
        pkv.testing_set_handoff_wait_ns(pkv.DEFAULT_HANDOFF_WAIT_NS)
    pkv.workspace_init(c.ws)
    compare_out(c.decode(), oracle_step(w)["out"])
    assert c.status() == 0


def test_handoff_limit_above_default_refused():
    with pytest.raises(pkv.PkvError):
        pkv.testing_set_handoff_wait_ns(pkv.DEFAULT_HANDOFF_WAIT_NS + 1)
