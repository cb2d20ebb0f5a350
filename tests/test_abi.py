"""C-ABI tests that need no GPU: the library loads, exports every symbol the
header declares, links no allocator, and its host-side planning and argument
checks behave as documented.  No case here reaches a kernel launch: every
negative case fails a host check first."""

import os
import re
import subprocess

import pytest

from paged_kv_gqa_16_gb300 import build as pkv_build
from paged_kv_gqa_16_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv_build.build()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:pkv|paged|decode)_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    declared = _declared_functions()
    assert set(declared) == set(pkv.EXPORTS)
    L = pkv.lib()
    for name in declared:
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for name in declared:
        assert re.search(rf"\bT {name}$", out, re.M), f"{name} not exported"


def test_links_no_device_allocator():
    out = subprocess.run(["nm", "-D", "--undefined-only", pkv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    bad = [l for l in out.splitlines() if re.search(r"cu(da)?Mem(Alloc|Free)|cudaMalloc|cudaFree", l)]
    assert not bad, bad


def test_version_and_strings():
    assert pkv.version() >> 16 == 1
    assert pkv.status_str(0) == "ok"
    assert "workspace" in pkv.status_str(pkv.PKV_ERR_WORKSPACE_TOO_SMALL)


def _d(**kw):
    base = dict(B=32, Hq=32, Hkv=8, D=128, page_size=16, num_pages=65536, num_indices=5000,
                max_seq_len=4096)
    base.update(kw)
    return pkv.dims(**base)


@pytest.mark.parametrize("max_len,S", [(4096, 1), (4096, 3), (4096, 7), (100, 8), (1, 1),
                                       (32768, 256), (0, 4)])
def test_split_chunk(max_len, S):
    d = _d(max_seq_len=max_len)
    c = pkv.split_chunk(d, S)
    assert c % 16 == 0 and c >= 16
    assert c * S >= max_len                      # the splits cover every token
    assert c - 16 < -(-max_len // S) or max_len == 0   # and are no coarser than needed


def test_workspace_layout_and_bytes():
    d = _d()
    for S in (1, 5, 64):
        ml, o = pkv.workspace_layout(d, S)
        n = d.B * d.Hq * S
        assert ml >= 256 + d.B * 8 and ml % 256 == 0 and o % 256 == 0
        assert o >= ml + n * 8
        assert pkv.workspace_bytes(d, S) >= o + n * d.D * 4
        assert pkv.workspace_bytes(d, S) % 256 == 0


@pytest.mark.parametrize("B,Hkv,max_len", [(1, 8, 32768), (32, 8, 4096), (8, 8, 1025),
                                            (128, 8, 8192), (1, 8, 16), (2, 2, 100)])
def test_plan_invariants(B, Hkv, max_len):
    d = _d(B=B, Hkv=Hkv, Hq=Hkv * 4, max_seq_len=max_len)
    S, ws = pkv.plan(d, num_sms=152)
    # persistent path: at most one block per SM, each with >= 64 tokens of capacity
    assert 1 <= S <= 152
    assert S <= max(1, -(-B * max_len // 64))
    assert ws == pkv.workspace_bytes(d, S)
    if B * max_len >= 152 * 64:
        assert S == 152


def test_plan_fallback_shape():
    # more than 4096 virtual rows: the per-(split, head, row) kernel is used
    d = _d(B=5000, Hq=2, Hkv=1, D=64, max_seq_len=4096)
    S, ws = pkv.plan(d, num_sms=152)
    assert 1 <= S <= -(-4096 // 256)
    assert ws == pkv.workspace_bytes(d, S)


def test_invalid_shapes_rejected():
    ws = 1 << 20
    fake = 1 << 32      # aligned, never dereferenced: every case fails a host check
    cases = [
        (_d(D=96), pkv.PKV_ERR_UNSUPPORTED),
        (_d(Hq=30), pkv.PKV_ERR_INVALID_ARG),
        (_d(Hq=8 * 17), pkv.PKV_ERR_UNSUPPORTED),
        (_d(page_size=0), pkv.PKV_ERR_INVALID_ARG),
        (_d(num_pages=0), pkv.PKV_ERR_INVALID_ARG),
        (_d(B=70000), pkv.PKV_ERR_INVALID_ARG),
        (_d(max_seq_len=-1), pkv.PKV_ERR_INVALID_ARG),
    ]
    for d, want in cases:
        with pytest.raises(pkv.PkvError) as e:
            pkv.lib()  # loaded
            code = pkv.lib().paged_decode_attn(pkv.ctypes.byref(d), fake, fake, fake, fake,
                                               fake, fake, 4, fake, ws, fake, None)
            pkv._check("paged_decode_attn", code)
        assert e.value.code == want, d


def test_argument_checks_before_launch():
    L = pkv.lib()
    d = _d()
    byref = pkv.ctypes.byref
    fake = 1 << 32
    # workspace too small
    need = pkv.workspace_bytes(d, 4)
    assert L.paged_decode_attn(byref(d), fake, fake, fake, fake, fake, fake, 4, fake, need - 1,
                               fake, None) == pkv.PKV_ERR_WORKSPACE_TOO_SMALL
    # misaligned pool / workspace / null out
    assert L.paged_decode_attn(byref(d), fake, fake + 2, fake, fake, fake, fake, 4, fake, need,
                               fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.paged_decode_attn(byref(d), fake, fake, fake, fake, fake, fake, 4, fake + 16, need,
                               fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.paged_decode_attn(byref(d), fake, fake, fake, fake, fake, fake, 4, fake, need,
                               None, None) == pkv.PKV_ERR_INVALID_ARG
    # split count out of range
    assert L.paged_decode_partials(byref(d), fake, fake, fake, fake, fake, fake, 0, fake, need,
                                   None) == pkv.PKV_ERR_INVALID_ARG
    # combine: null partials
    assert L.decode_combine(byref(d), None, fake, 4, fake, None) == pkv.PKV_ERR_INVALID_ARG
    # append: rope table given with no rows, misaligned k_new, rope_q without q
    assert L.paged_kv_append(byref(d), fake, fake, fake, fake, fake, fake, fake, fake, fake, 0,
                             0, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.paged_kv_append(byref(d), fake, fake + 8, fake, fake, fake, fake, fake, fake, None,
                             0, 0, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert L.paged_kv_append(byref(d), None, fake, fake, fake, fake, fake, fake, fake, fake,
                             16, 1, None, None) == pkv.PKV_ERR_INVALID_ARG
    # rope table: odd D
    assert L.pkv_rope_table(fake, 16, 63, 10000.0, None) == pkv.PKV_ERR_INVALID_ARG
    # workspace init: misaligned
    assert L.pkv_workspace_init(fake + 4, 4096, None) == pkv.PKV_ERR_INVALID_ARG
    # B = 0 is a valid no-op that launches nothing
    d0 = _d(B=0)
    assert L.paged_decode_attn(byref(d0), None, None, None, None, None, None, 4, None, 0, None,
                               None) == pkv.PKV_OK


def test_advance_argument_checks():
    L = pkv.lib()
    d = _d(B=4)
    byref = pkv.ctypes.byref
    fake = 1 << 32
    ok_args = dict(seq_lens=fake, ptr=fake, ind=fake, free=fake, n_free=8, head=fake, st=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return L.paged_kv_advance(byref(d), a["seq_lens"], a["ptr"], a["ind"], a["free"],
                                  a["n_free"], a["head"], a["st"], None)

    assert call(seq_lens=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(ptr=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(head=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(n_free=-1) == pkv.PKV_ERR_INVALID_ARG
    assert call(free=None) == pkv.PKV_ERR_INVALID_ARG          # num_free > 0 needs a list
    assert call(seq_lens=fake + 2) == pkv.PKV_ERR_INVALID_ARG  # misaligned
    assert call(st=fake + 1) == pkv.PKV_ERR_INVALID_ARG
    d0 = _d(B=0)
    assert L.paged_kv_advance(byref(d0), None, None, None, None, 0, None, None,
                              None) == pkv.PKV_OK


def test_step_advance_argument_checks():
    """The advance's arguments are checked before anything is launched."""
    L = pkv.lib()
    byref = pkv.ctypes.byref
    fake = 1 << 32
    d = _d(B=4)
    S = 2
    wsb = pkv.workspace_bytes(d, S)

    def call(d=d, **kw):
        a = dict(q=fake, kn=fake, vn=fake, k=fake, v=fake, ind=fake, ptr=fake, sl=fake,
                 rope=None, ws=fake, out=fake, free=fake, n_free=8, head=fake)
        a.update(kw)
        return L.paged_decode_step_advance(
            byref(d), a["q"], a["kn"], a["vn"], a["k"], a["v"], a["ind"], a["ptr"], a["sl"],
            a["rope"], 0, S, a["ws"], wsb, a["out"], a["free"], a["n_free"], a["head"], None)

    assert call(head=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(n_free=-1) == pkv.PKV_ERR_INVALID_ARG
    assert call(free=None) == pkv.PKV_ERR_INVALID_ARG            # num_free > 0 needs a list
    assert call(head=fake + 2) == pkv.PKV_ERR_INVALID_ARG        # misaligned
    assert call(kn=None) == pkv.PKV_ERR_INVALID_ARG              # the step's own checks
    assert call(ws=fake + 16) == pkv.PKV_ERR_INVALID_ARG
    assert call(d=_d(B=0), head=None, free=None, n_free=0) == pkv.PKV_OK


def test_prefill_argument_checks():
    L = pkv.lib()
    byref = pkv.ctypes.byref
    fake = 1 << 32

    def call(d, total_q=16, max_q=16, **kw):
        a = dict(q=fake, qo=fake, k=fake, v=fake, ind=fake, ptr=fake, sl=fake, out=fake, st=None)
        a.update(kw)
        return L.paged_prefill_attn(byref(d), a["q"], a["qo"], total_q, max_q, a["k"], a["v"],
                                    a["ind"], a["ptr"], a["sl"], a["out"], a["st"], None)

    d = _d(B=4)
    assert call(_d(B=4, scale=0.0)) == pkv.PKV_ERR_INVALID_ARG      # the scale must be > 0
    assert call(d, total_q=-1) == pkv.PKV_ERR_INVALID_ARG
    assert call(d, max_q=-1) == pkv.PKV_ERR_INVALID_ARG
    assert call(d, q=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(d, out=fake + 8) == pkv.PKV_ERR_INVALID_ARG          # misaligned
    assert call(d, qo=fake + 2) == pkv.PKV_ERR_INVALID_ARG
    assert call(_d(B=70000 // 8, Hkv=8)) == pkv.PKV_ERR_UNSUPPORTED  # B * Hkv > 65535
    assert call(d, total_q=0) == pkv.PKV_OK                           # nothing to do


def test_plan_argument_checks():
    """paged_decode_plan refuses bad arguments on the host, before any launch."""
    import ctypes
    L = pkv.lib()
    d = _d()
    S = 8
    need = pkv.workspace_bytes(d, S)
    fake = 1 << 32
    # num_splits out of range
    assert L.paged_decode_plan(ctypes.byref(d), fake, fake, fake, 0, fake, need, None) == \
        pkv.PKV_ERR_INVALID_ARG
    # no workspace, or one too small
    assert L.paged_decode_plan(ctypes.byref(d), fake, fake, fake, S, None, need, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert L.paged_decode_plan(ctypes.byref(d), fake, fake, fake, S, fake, need - 256, None) == \
        pkv.PKV_ERR_WORKSPACE_TOO_SMALL
    # a misaligned workspace
    assert L.paged_decode_plan(ctypes.byref(d), fake, fake, fake, S, fake + 16, need, None) == \
        pkv.PKV_ERR_INVALID_ARG
    # an empty batch needs no plan
    d0 = _d(B=0)
    assert L.paged_decode_plan(ctypes.byref(d0), None, None, None, S, None, 0, None) == pkv.PKV_OK


def test_workspace_holds_the_plan():
    """The workspace grows with the plan: one 72-word entry per block."""
    d = _d()
    assert pkv.workspace_bytes(d, 152) - pkv.workspace_bytes(d, 8) >= 144 * 72 * 4


def test_prefill_workspace_bytes():
    """Per SM a slot of two tiles x 128 rows: D bf16 and an fp32 (base, l)
    pair each; 0 for an unbuilt head dim or SM count."""
    assert pkv.prefill_workspace_bytes(128, 152) == 152 * 2 * 128 * (128 * 2 + 8)
    assert pkv.prefill_workspace_bytes(64, 152) == 152 * 2 * 128 * (64 * 2 + 8)
    assert pkv.prefill_workspace_bytes(64, 1) == 2 * 128 * (64 * 2 + 8)
    # the rows of any number of slots end on a 256-byte boundary
    assert (2 * 128 * 128 * 2) % 256 == 0 and (2 * 128 * 64 * 2) % 256 == 0
    for D, n in [(96, 152), (256, 152), (128, 0), (128, -3), (64, 1025)]:
        assert pkv.prefill_workspace_bytes(D, n) == 0


def _pd(B, Hq, Hkv, D, max_seq_len=8192):
    return pkv.dims(B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=16, num_pages=100000,
                    num_indices=100000, max_seq_len=max_seq_len)


def test_prefill_plan_bench_shapes():
    """The list paged_prefill_attn(_ws) launches on 152 SMs for the three
    bench shapes: the extend's 512 equal units leave a last round of 56, cut
    in two with a workspace; the causal prefills are pair-major lists of many
    rounds and are never cut."""
    ws128 = pkv.prefill_workspace_bytes(128, 152)
    ext = _pd(16, 32, 8, 128)
    assert pkv.prefill_plan(ext, 256, 152) == dict(
        pairs=4, units=512, group_rows=38, entries=512, split=1, split_base=512, grid=152)
    assert pkv.prefill_plan(ext, 256, 152, ws128) == dict(
        pairs=4, units=512, group_rows=38, entries=456 + 112, split=2, split_base=456, grid=152)
    # 4 x 4096 at n_rep 4: 128 tiles of 32 tokens, 64 pairs, 2,048 units
    p = pkv.prefill_plan(_pd(4, 32, 8, 128), 4096, 152, ws128)
    assert p == dict(pairs=64, units=2048, group_rows=32, entries=2048, split=1,
                     split_base=2048, grid=152)
    p = pkv.prefill_plan(_pd(32, 32, 8, 64), 512, 152, pkv.prefill_workspace_bytes(64, 152))
    assert p["units"] == 2048 and p["split"] == 1 and p["group_rows"] == 256


def test_prefill_plan_split_rules():
    ws = lambda n: pkv.prefill_workspace_bytes(128, n)
    # one round (38 units of one 1,200-token row): every unit cut, 152 / 38 = 4
    p = pkv.prefill_plan(_pd(1, 8, 2, 128), 1200, 152, ws(152))
    assert (p["units"], p["split"], p["split_base"], p["entries"], p["grid"]) == (38, 4, 0, 152, 152)
    # at most 16 parts a unit
    p = pkv.prefill_plan(_pd(1, 8, 2, 128), 60, 152, ws(152))
    assert (p["units"], p["split"], p["entries"]) == (2, 16, 32)
    # the workspace's slots bound the parts: 5 slots for 2 units -> 2 each; 3 -> none
    assert pkv.prefill_plan(_pd(1, 8, 2, 128), 60, 152, ws(5))["split"] == 2
    assert pkv.prefill_plan(_pd(1, 8, 2, 128), 60, 152, ws(3))["split"] == 1
    # a last round of more than half the SMs is not cut: 229 units, 77 in the last
    p = pkv.prefill_plan(_pd(229, 16, 1, 128), 8, 152, ws(152))
    assert (p["units"], p["split"]) == (229, 1)
    p = pkv.prefill_plan(_pd(228, 16, 1, 128), 8, 152, ws(152))
    assert (p["units"], p["split"], p["split_base"], p["entries"]) == (228, 2, 152, 304)
    # a pair-major list of several rounds (chunks of more than 4 pairs) is not cut
    p = pkv.prefill_plan(_pd(1, 32, 8, 128), 320, 152, ws(152))      # 5 pairs, 40 units
    assert (p["pairs"], p["units"], p["split"]) == (5, 40, 3)        # one round: cut
    p = pkv.prefill_plan(_pd(4, 32, 8, 128), 320, 152, ws(152))      # 160 units, 2 rounds
    assert (p["pairs"], p["units"], p["split"]) == (5, 160, 1)
    # nothing to run
    assert pkv.prefill_plan(_pd(2, 8, 2, 128), 0, 152, ws(152))["units"] == 0


def test_prefill_plan_rejects():
    d = _pd(2, 8, 2, 128)
    for args in [(-1, 152), (16, 0), (16, 1025)]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.prefill_plan(d, *args)
        assert e.value.code == pkv.PKV_ERR_INVALID_ARG
