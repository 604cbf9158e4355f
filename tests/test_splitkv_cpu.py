"""Split-KV host logic: the split-count heuristic, workspace sizes and
argument checks (no CUDA call)."""
import math

import pytest


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


TASK_COST = 5  # fixed start-up of a key range, in K/V block times


def cost(units, kvb, s, sms):
    """Modelled time of s ranges: waves of tasks times (blocks per range + start-up)."""
    bps = math.ceil(kvb / s)
    tasks = units * math.ceil(kvb / bps)
    return math.ceil(tasks / sms) * (bps + TASK_COST)


@pytest.mark.parametrize("shape", [
    # B, Hq, Hkv, Sq, Sk, causal
    (8, 32, 8, 1, 32768, 0), (32, 32, 1, 1, 16384, 0), (8, 32, 8, 4, 16384, 1), (1, 8, 8, 1, 4096, 0),
    (2, 16, 2, 1, 100000, 0), (1, 1, 1, 1, 1024, 0), (3, 8, 2, 1, 1000, 0), (4, 32, 8, 1, 16384, 0),
])
def test_heuristic(fa, shape):
    B, Hq, Hkv, Sq, Sk, causal = shape
    sms = 152
    s = fa.fa_splitkv_num_splits(B, Hq, Hkv, Sq, Sk, 128, 128, causal, sms)
    plan = fa.fa_make_plan(B, Hq, Hkv, Sq, Sk, 128, 128, causal)
    units = B * plan.groups * plan.mblocks
    kvb = plan.kv_blocks
    if units >= sms or kvb < 8:
        assert s == 1
        return
    assert 1 <= s <= min(128, kvb // 4)
    assert math.ceil(kvb / math.ceil(kvb / s)) == s  # no empty range
    counts = range(1, min(128, kvb // 4) + 1)
    best = min(cost(units, kvb, t, sms) for t in counts)
    assert cost(units, kvb, s, sms) == best
    assert all(cost(units, kvb, t, sms) > best for t in counts if math.ceil(kvb / math.ceil(kvb / t)) < s)


def test_decode_choices(fa):
    # measured best counts on GB300 (TFLOP/s and GB/s sweeps over 1..32 ranges)
    assert fa.fa_splitkv_num_splits(8, 32, 8, 1, 32768, 128, 128, 0, 152) == 7   # decode32k: 448 tasks, 3 waves
    assert fa.fa_splitkv_num_splits(32, 32, 1, 1, 16384, 128, 128, 0, 152) == 4  # MQA decode: one wave of 128
    assert fa.fa_splitkv_num_splits(8, 32, 8, 4, 16384, 128, 128, 1, 152) == 2   # 4 draft tokens: one wave
    assert fa.fa_splitkv_num_splits(64, 32, 8, 1, 32768, 128, 128, 0, 152) == 1  # 512 tasks already


def test_workspace_size(fa):
    assert fa.fa_splitkv_workspace_size(8, 32, 1, 128, 7) == 7 * 8 * 32 * 129 * 4
    assert fa.fa_splitkv_workspace_size(8, 32, 1, 128, 1) == 0
    assert fa.fa_splitkv_workspace_size(8, 32, 1, 128, 0) == 0


FAKE = 0x10000


def test_argument_checks(fa):
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 1, 1000, 128, 128, 0, 0.0)
    assert fa.fa_fwd_splitkv(*args, -1, FAKE, 1 << 20, None) == 1
    assert fa.fa_fwd_splitkv(*args, 1025, FAKE, 1 << 20, None) == 1
    assert fa.fa_fwd_splitkv(*args, 4, FAKE + 4, 1 << 20, None) == 1
    o = fa.default_options()
    o.exp_emu = 1
    assert fa.fa_fwd_splitkv(*args, 4, FAKE, 1 << 20, None, o) == 2
    o = fa.default_options()
    o.workspace = FAKE
    assert fa.fa_fwd_splitkv(*args, 4, FAKE, 1 << 20, None, o) == 2
    # empty problems need no pointer
    assert fa.fa_fwd_splitkv(None, None, None, None, None, 0, 8, 2, 1, 1000, 128, 128, 0, 0.0, 4, None, 0,
                             None) == 0
