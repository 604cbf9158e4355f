"""Host-only checks of the C ABI (no GPU needed): exports, argument validation
and the tile plan the kernel runs."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = _declared_functions()
    for required in ("fa_fwd", "fa_fwd_ex", "fa_device_status", "fa_device_status_detail", "fa_status_string",
                     "fa_make_plan",
                     "fa_plan_task", "fa_options_default", "fa_version", "fa_plan_block_masked",
                     "fa_selftest_exp2", "fa_plan_first_masked_block", "fa_fwd_varlen", "fa_fwd_varlen_ex",
                     "fa_varlen_workspace_size", "fa_varlen_plan_host"):
        assert required in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(fa):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(4) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"
    assert fa.fa_version() >= 100


BASE = dict(batch=1, heads_q=4, heads_kv=2, seqlen_q=64, seqlen_k=64, d_qk=128, d_v=128, causal=0, scale=0.0)
FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced by these cases


def _call(fa, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, **kw):
    a = dict(BASE)
    a.update(kw)
    return fa.fa_fwd(q, k, v, o, lse, a["batch"], a["heads_q"], a["heads_kv"], a["seqlen_q"], a["seqlen_k"],
                     a["d_qk"], a["d_v"], a["causal"], a["scale"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1),
    (dict(heads_q=6, heads_kv=4), 1), (dict(heads_kv=0), 1), (dict(heads_q=0), 1), (dict(batch=-1), 1),
    (dict(seqlen_q=-5), 1), (dict(seqlen_k=-1), 1), (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1), (dict(scale=-0.5), 1), (dict(q=FAKE + 8), 1), (dict(lse=FAKE + 4), 1),
    (dict(d_qk=96, d_v=96), 2), (dict(d_qk=64, d_v=128), 2), (dict(d_qk=256, d_v=128), 2),
    (dict(d_qk=128, d_v=32), 2),
])
def test_invalid_arguments_rejected_before_cuda(fa, kw, code):
    assert _call(fa, **kw) == code


@pytest.mark.parametrize("kw", [dict(batch=0), dict(seqlen_q=0)])
def test_empty_problem_is_ok_without_launch(fa, kw):
    # null pointers are fine: nothing is touched
    assert _call(fa, q=None, k=None, v=None, o=None, lse=None, **kw) == 0


def test_bad_options_rejected(fa):
    opts = fa.default_options()
    assert abs(opts.tau - 8.0) < 1e-7 and opts.pack == 0 and opts.grid == 0 and opts.no_balance == 0
    for field, value in (("pack", 3), ("pack", -1), ("grid", -2), ("debug_flags", 16), ("debug_flags", 8),
                         ("timeout_s", 1e9), ("tau", 65.0), ("tau", float("inf")), ("tau", float("nan")), ("exp_emu", 2),
                         ("exp_emu", -1), ("store_mode", 3), ("store_mode", -1), ("no_balance", 2),
                         ("no_balance", -1)):
        o = fa.default_options()
        setattr(o, field, value)
        rc = fa.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 64, 128, 128, 0, 0.0, o, None)
        assert rc == 1, (field, value)


VBASE = dict(batch=2, total_q=300, total_k=400, heads_q=4, heads_kv=2, d_qk=128, d_v=128, causal=1, scale=0.0)


def _vcall(fa, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, cu_q=FAKE, cu_k=FAKE, ws=FAKE, ws_bytes=None, opts=None,
           **kw):
    a = dict(VBASE)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = fa.fa_varlen_workspace_size(max(a["batch"], 0), max(a["heads_q"], 1), max(a["total_q"], 0))
    return fa.fa_fwd_varlen_ex(q, k, v, o, lse, cu_q, cu_k, a["batch"], a["total_q"], a["total_k"], a["heads_q"],
                               a["heads_kv"], a["d_qk"], a["d_v"], a["causal"], a["scale"], ws, ws_bytes, opts, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(k=None), 1), (dict(cu_q=None), 1), (dict(cu_k=None), 1),
    (dict(ws=None), 1), (dict(ws=FAKE + 8), 1), (dict(cu_q=FAKE + 2), 1), (dict(q=FAKE + 8), 1),
    (dict(batch=-1), 1), (dict(batch=16385), 1), (dict(total_q=-1), 1), (dict(total_k=-3), 1),
    (dict(total_q=2 ** 30, total_k=2 ** 30), 1), (dict(heads_q=6, heads_kv=4), 1), (dict(scale=-1.0), 1),
    (dict(d_qk=96, d_v=96), 2), (dict(d_qk=64, d_v=128), 2),
])
def test_varlen_invalid_arguments_rejected_before_cuda(fa, kw, code):
    assert _vcall(fa, **kw) == code


def test_sched_workspace_options(fa):
    o = fa.default_options()
    assert o.workspace is None
    o.workspace = FAKE + 8  # misaligned
    assert fa.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 64, 128, 128, 1, 0.0, o, None) == 1
    o.workspace = FAKE
    o.exp_emu = 1  # one or the other
    assert fa.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 64, 128, 128, 1, 0.0, o, None) == 2
    o = fa.default_options()
    o.workspace = FAKE  # varlen calls take their own workspace
    assert _vcall(fa, opts=o) == 1


def test_varlen_workspace_too_small_and_exp_emu(fa):
    need = fa.fa_varlen_workspace_size(2, 4, 300)
    assert need == 256 + 32 * 4 * ((300 + 255) // 256 + 2)
    assert _vcall(fa, ws_bytes=need - 1) == 1
    o = fa.default_options()
    o.exp_emu = 1
    assert _vcall(fa, opts=o) == 2
    assert fa.fa_varlen_workspace_size(-1, 4, 10) == 0


@pytest.mark.parametrize("kw", [dict(batch=0), dict(total_q=0)])
def test_varlen_empty_is_ok_without_launch(fa, kw):
    assert _vcall(fa, q=None, k=None, v=None, o=None, lse=None, cu_q=None, cu_k=None, ws=None, ws_bytes=0,
                  **kw) == 0


# ---------------------------------------------------------------------------
# the tile plan
# ---------------------------------------------------------------------------

PLAN_CASES = [
    # B, Hq, Hkv, Sq, Sk, dq, dv, causal
    (1, 1, 1, 128, 128, 64, 64, 0),
    (2, 4, 4, 300, 300, 128, 128, 0),
    (2, 4, 4, 300, 300, 128, 128, 1),
    (1, 8, 2, 200, 456, 128, 128, 1),
    (1, 8, 2, 456, 200, 128, 128, 1),   # rows with no visible key
    (2, 32, 8, 1000, 1000, 128, 128, 1),
    (1, 32, 1, 513, 513, 128, 128, 1),  # MQA, ratio 32
    (1, 6, 2, 77, 77, 192, 128, 1),     # ratio 3: one head per tile
    (1, 256, 1, 20, 40, 64, 64, 0),     # ratio 256 > 128
    (3, 2, 2, 1, 1, 64, 64, 1),
    (1, 2, 1, 129, 1, 128, 64, 1),
]


def _visible_last(Sq, Sk, causal, pos):
    return Sk - 1 if not causal else min(Sk - 1, pos + Sk - Sq)


@pytest.mark.parametrize("case", PLAN_CASES, ids=lambda c: "x".join(map(str, c)))
def test_plan_covers_every_row_once_with_exact_block_counts(fa, case):
    B, Hq, Hkv, Sq, Sk, dq, dv, causal = case
    plan = fa.fa_make_plan(B, Hq, Hkv, Sq, Sk, dq, dv, causal, l2_bytes=1 << 20)
    ratio = Hq // Hkv
    assert plan.pack == (ratio if 128 % ratio == 0 else 1)
    assert plan.groups * plan.pack == Hq and plan.pos_per_tile * plan.pack == 128
    seen = np.zeros((B, Hq, Sq), dtype=np.int32)
    costs = []
    for t in range(plan.num_tasks):
        task = fa.fa_plan_task(plan, t)
        assert task.kv_head == (task.g * plan.pack) // ratio
        nmax = 0
        for s in range(2):
            pos0, n = task.pos0[s], task.n_blocks[s]
            rows = np.arange(128)
            pos = pos0 + rows // plan.pack
            head = task.g * plan.pack + rows % plan.pack
            ok = pos < Sq
            assert np.all(head // ratio == task.kv_head)
            np.add.at(seen, (task.b, head[ok], pos[ok]), 1)
            # brute-force block count: blocks holding a key visible to some row
            lasts = [_visible_last(Sq, Sk, causal, int(p)) for p in pos[ok]]
            want = 0 if not lasts or max(lasts) < 0 else max(lasts) // 128 + 1
            assert n == want, (t, s, n, want)
            # a block without the mask flag must be fully visible to every row
            for j in range(n):
                if not fa.fa_plan_block_masked(plan, pos0, j):
                    assert (j + 1) * 128 <= Sk and all(l >= j * 128 + 127 for l in lasts)
            nmax = max(nmax, n)
        costs.append(nmax)
    assert np.all(seen == 1)
    if causal:
        # longest first: inside each L2 section of the heavier half, then over
        # the whole lighter half; every heavy task costs at least every light one
        units = B * plan.groups
        nh = units * plan.heavy_levels
        assert plan.heavy_levels == (plan.mblocks + 1) // 2
        per_section = plan.section_units * plan.heavy_levels
        for s0 in range(0, nh, per_section):
            c = costs[s0:min(s0 + per_section, nh)]
            assert all(a >= b for a, b in zip(c, c[1:]))
        light = costs[nh:]
        assert all(a >= b for a, b in zip(light, light[1:]))
        if light:
            assert min(costs[:nh]) >= max(light)


def test_plan_sections_follow_l2_budget(fa):
    # 16 heads of S=32k, d=128: K+V per head = 32768 * 256 * 2 = 16 MiB
    plan = fa.fa_make_plan(1, 16, 16, 32768, 32768, 128, 128, 1, l2_bytes=64 << 20)
    assert plan.section_units == 4
    plan = fa.fa_make_plan(1, 16, 16, 32768, 32768, 128, 128, 1, l2_bytes=1)
    assert plan.section_units == 1


def test_plan_default_section_budget_is_8_mib(fa):
    """Without an explicit budget the plan sizes causal sections as the launch
    does on a large L2: about 8 MiB of K/V per section."""
    # causal 1k, 32 x 16 heads: K+V per (b, head) = 1024 * 256 * 2 B = 512 KiB -> 16 units
    plan = fa.fa_make_plan(32, 16, 16, 1024, 1024, 128, 128, 1)
    assert plan.section_units == 16
    # causal 8k, 4 x 16: 4 MiB per unit -> 2 units
    plan = fa.fa_make_plan(4, 16, 16, 8192, 8192, 128, 128, 1)
    assert plan.section_units == 2
    # more K/V per unit than the budget: one unit per section
    plan = fa.fa_make_plan(1, 16, 16, 32768, 32768, 128, 128, 1)
    assert plan.section_units == 1


def test_plan_rejects_bad_pack(fa):
    with pytest.raises(fa.FaError):
        fa.fa_make_plan(1, 8, 2, 64, 64, 128, 128, 0, pack=3)
    plan = fa.fa_make_plan(1, 8, 2, 64, 64, 128, 128, 0, pack=1)
    assert plan.pack == 1 and plan.groups == 8
