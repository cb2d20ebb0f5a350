"""The per-step plan (paged_decode_plan) and the planned calls, on the GPU
through the C ABI.  A planned call runs the same partition as the unplanned
one, so its output is the same bit for bit; both match the fp64 oracle.
Also: one plan serving several calls (the layers of a step) inside one CUDA
graph, a plan made for another grid (the call falls back to computing the
partition), a plan left over from longer rows (no fault; a new plan restores
the result), and the plan's own length checks."""

import numpy as np
import pytest
import torch

from gpu_cases import GpuCase, bits, compare_out, oracle_step
from paged_kv_gqa_16_gb300 import pkv
from paged_kv_gqa_16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _plan(c, S=None):
    t = c.t
    pkv.paged_decode_plan(c.d, t["kv_indices"], t["kv_indptr"], t["seq_lens"],
                          c.S if S is None else S, c.ws)


def _attn(c, planned, S=None):
    t = c.t
    out = torch.empty_like(c.out)
    fn = pkv.paged_decode_attn_planned if planned else pkv.paged_decode_attn
    fn(c.d, t["q"], t["k_pool"], t["v_pool"], t["kv_indices"], t["kv_indptr"], t["seq_lens"],
       c.S if S is None else S, c.ws, out)
    return out


def _step(c, planned, k_pool, v_pool):
    t = c.t
    out = torch.empty_like(c.out)
    fn = pkv.paged_decode_step_planned if planned else pkv.paged_decode_step
    fn(c.d, t["q"], t["k_new"], t["v_new"], k_pool, v_pool, t["kv_indices"], t["kv_indptr"],
       t["seq_lens"], c.rope, c.rope_max_pos, c.S, c.ws, out)
    return out


@pytest.mark.parametrize("name", ["tiny", "gqa_1b", "ragged_b32", "long_32k", "serving_b1",
                                  "serving_b4", "serving_b32", "serving_b128"])
def test_planned_equals_unplanned_and_oracle(name):
    w = wl.make(name)
    c = GpuCase(w)
    t = c.t
    kp0, vp0 = t["k_pool"].clone(), t["v_pool"].clone()
    # the whole step: planned and unplanned from the same pools
    want = _step(c, False, t["k_pool"], t["v_pool"]).clone()
    kp_a, vp_a = t["k_pool"].clone(), t["v_pool"].clone()
    t["k_pool"].copy_(kp0)
    t["v_pool"].copy_(vp0)
    _plan(c)
    got = _step(c, True, t["k_pool"], t["v_pool"])
    torch.cuda.synchronize()
    assert c.status() == 0
    assert np.array_equal(bits(got), bits(want))
    assert np.array_equal(bits(t["k_pool"]), bits(kp_a))
    assert np.array_equal(bits(t["v_pool"]), bits(vp_a))
    compare_out(got, oracle_step(w)["out"])
    # attention alone over the appended pools, on the same plan
    a0 = _attn(c, False)
    a1 = _attn(c, True)
    torch.cuda.synchronize()
    assert np.array_equal(bits(a0), bits(a1))


def test_one_plan_many_layers_in_a_graph():
    """A step of four layers (here: four queries over one pool): one plan,
    then each layer's planned call, captured in one graph.  Replayed after
    new lengths are written in place, the plan inside the graph follows them;
    every layer matches its unplanned call bit for bit."""
    w = wl.make("gqa_1b")
    c = GpuCase(w)
    c.append()                           # the new token's slot, as in a step
    t = c.t
    g_ = torch.Generator().manual_seed(7)
    qs = [torch.randn(t["q"].shape, generator=g_).to(torch.bfloat16).cuda() for _ in range(4)]
    outs = [torch.empty_like(c.out) for _ in qs]

    def run():
        pkv.paged_decode_plan(c.d, t["kv_indices"], t["kv_indptr"], t["seq_lens"], c.S, c.ws)
        for q, o in zip(qs, outs):
            pkv.paged_decode_attn_planned(c.d, q, t["k_pool"], t["v_pool"], t["kv_indices"],
                                          t["kv_indptr"], t["seq_lens"], c.S, c.ws, o)

    run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    lens0 = t["seq_lens"].clone()
    # the same pages, each row 1..300 tokens shorter: every slot still valid
    shorter = (lens0 - torch.randint(1, 301, lens0.shape, generator=g_).to(lens0)).clamp(min=1)
    for lens in (lens0, shorter):
        t["seq_lens"].copy_(lens)
        graph.replay()
        torch.cuda.synchronize()
        assert pkv.status_word(c.ws) == 0
        for q, o in zip(qs, outs):
            ref = torch.empty_like(c.out)
            pkv.paged_decode_attn(c.d, q, t["k_pool"], t["v_pool"], t["kv_indices"],
                                  t["kv_indptr"], t["seq_lens"], c.S, c.ws, ref)
            torch.cuda.synchronize()
            assert np.array_equal(bits(o), bits(ref))


def test_plan_for_another_grid_falls_back():
    w = wl.make("ragged_b32")
    c = GpuCase(w, num_splits=152)
    c.append()
    want = _attn(c, False, S=100).clone()
    _plan(c, S=152)                      # a plan for 152 blocks ...
    got = _attn(c, True, S=100)          # ... used by a call of 100
    torch.cuda.synchronize()
    assert c.status() == 0
    assert np.array_equal(bits(got), bits(want))


def test_plan_left_from_longer_rows_then_replanned():
    """The caller shortens every row without planning again: the planned
    call reads only pages the table still names (no fault, status clean);
    after a new plan it matches the unplanned call bit for bit."""
    w = wl.build("stale", B=6, Hq=32, Hkv=8, D=128, page_size=16,
                 seq_lens=[900, 40, 1500, 700, 33, 1200], seed=4, fill_new_slot=True)
    c = GpuCase(w)
    _plan(c)
    c.t["seq_lens"].copy_(torch.tensor([500, 20, 1000, 100, 17, 600], dtype=torch.int32))
    _attn(c, True)
    torch.cuda.synchronize()
    assert c.status() == 0
    _plan(c)
    got = _attn(c, True)
    want = _attn(c, False)
    torch.cuda.synchronize()
    assert np.array_equal(bits(got), bits(want))


def test_plan_sets_length_flag():
    w = wl.build("pflag", B=3, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[20, 40, 5], seed=2)
    c = GpuCase(w, num_splits=2)
    c.t["seq_lens"][0] = w.max_seq_len + 1
    _plan(c)
    assert c.status() & pkv.FLAG_BAD_LEN


@pytest.mark.parametrize("name", ["gqa_1b", "long_32k", "serving_b64"])
def test_unplanned_call_leaves_the_plan(name):
    """The first call of a step (unplanned) leaves its partition in the
    workspace; the step's later calls run on it without paged_decode_plan,
    bit for bit the same as unplanned calls."""
    w = wl.make(name)
    c = GpuCase(w)
    c.append()
    first = _attn(c, False).clone()          # writes the plan
    later = _attn(c, True)                   # runs on it
    torch.cuda.synchronize()
    assert c.status() == 0
    assert np.array_equal(bits(first), bits(later))
    compare_out(later, oracle_step(w)["out"])
