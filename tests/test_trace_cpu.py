"""The event-log reader on a hand-made buffer (no GPU): record layout, clock
unwrapping across the 32-bit wrap, per-track order, and the intervals the
summary reports.  Also the ABI's early rejection of bad trace options."""
import numpy as np
import pytest

from exact_attention_forward_08_gb300 import trace as tr


def rec(code, arg, clock):
    return (tr.CODES[code] << 56) | ((arg & 0xFFFFFF) << 32) | (clock & 0xFFFFFFFF)


def buffer(tracks, cap=64):
    """tracks: dict track name -> list of (event, arg, clock) for one CTA."""
    words = np.zeros(tr.trace_words(1, cap), dtype=np.uint64)
    for k, name in enumerate(tr.TRACKS):
        evs = tracks.get(name, [])
        base = k * (cap + 1)
        words[base] = len(evs)
        for i, (ev, arg, clk) in enumerate(evs):
            words[base + 1 + i] = rec(ev, arg, clk)
    return words


def one_block_log(t0):
    """Stage 0, blocks 0 and 1 of one task, starting at clock t0 (may wrap)."""
    sm = []
    mm = [("mm_task", 0, t0), ("mm_qk", 0, t0 + 10)]
    for j, base in ((0, t0 + 100), (1, t0 + 3100)):
        sm += [("sm_wait", j, base), ("sm_s", j, base + 500), ("sm_p", j, base + 1550)]
        mm += [("mm_p", j, base + 1700), ("mm_pv", j, base + 2200)]
        if j == 0:
            mm += [("mm_qk", 1, base + 2800)]
    return {"softmax0": [("sm_task", 0, t0 + 1)] + sm, "mma": mm}


@pytest.mark.parametrize("t0", [1000, (1 << 32) - 2000])
def test_decode_and_intervals(t0):
    log = one_block_log(t0)
    dec = tr.decode(buffer(log), 1, 64)
    assert len(dec) == 1
    cta = dec[0]
    assert cta["_counts"]["softmax0"] == 7 and cta["_counts"]["mma"] == 7
    times = [t for t, _, _ in cta["softmax0"]]
    assert times == sorted(times) and times[0] == 1  # relative to the first event (mm_task at t0)
    assert [e for _, e, _ in cta["mma"]][:2] == ["mm_task", "mm_qk"]
    s = tr.summarize(dec)
    assert s["softmax.steady.wait_for_S"]["median"] == 500
    assert s["softmax.steady.work_S_to_P"]["median"] == 1050
    assert s["mma.issue_PV"]["median"] == 500
    assert s["handoff.softmax_P_to_mma_P.steady"]["median"] == 150
    # S of block 1 at t0 + 3600, its Q K^T issued at t0 + 2900
    assert s["handoff.QK_issue_to_softmax_S.steady"]["median"] == 700
    assert s["stage.block_period"]["median"] == 3000


def test_records_past_cap_are_counted_not_kept():
    cap = 4
    words = np.zeros(tr.trace_words(1, cap), dtype=np.uint64)
    words[0] = 9  # the kernel counted 9 records on track 0
    for i in range(cap):
        words[1 + i] = rec("sm_s", i, 100 * i)
    dec = tr.decode(words, 1, cap)
    assert dec[0]["_counts"]["softmax0"] == 9
    assert len(dec[0]["softmax0"]) == cap


def test_abi_rejects_bad_trace_options_before_cuda():
    import exact_attention_forward_08_gb300 as fa
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    fa.load_library()
    fake = 0x10000
    for ctas, cap, ptr in ((0, 10, fake), (1, 0, fake), (1, 10, fake + 4)):
        o = fa.default_options()
        o.trace, o.trace_ctas, o.trace_cap = ptr, ctas, cap
        rc = fa.fa_fwd_ex(fake, fake, fake, fake, fake, 1, 2, 2, 128, 128, 128, 128, 0, 0.0, o, None)
        assert rc == fa.FA_ERR_INVALID_ARG
    o = fa.default_options()
    o.debug_flags = fa.DEBUG_PLANT_BAD_TASK  # only together with DEBUG_CHECKS
    assert fa.fa_fwd_ex(fake, fake, fake, fake, fake, 1, 2, 2, 128, 128, 128, 128, 0, 0.0, o, None) == \
        fa.FA_ERR_INVALID_ARG
    o.debug_flags = 16  # unknown bit
    assert fa.fa_fwd_ex(fake, fake, fake, fake, fake, 1, 2, 2, 128, 128, 128, 128, 0, 0.0, o, None) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_status_string(5) == "FA_ERR_DEVICE_CHECK"


def test_backward_intervals():
    """Two streamed blocks of one task on stage 0 of the backward log."""
    row = [("br_task", 0, 0)]
    mma = [("bm_task", 0, 5), ("bm_t", 0, 10), ("bm_sdp", 0, 400)]
    tma = [("bl_task", 0, 0), ("bl_t", 0, 2), ("bl_t", 1, 3), ("bl_t", 2, 1000)]
    for it, base in ((0, 100), (1, 3100)):
        row += [("br_wait", it, base), ("br_s", it, base + 600), ("br_p", it, base + 1900)]
        mma += [("bm_p", it, base + 2000), ("bm_acc", it, base + 2600)]
        if it == 0:
            mma += [("bm_t", 1, base + 2700), ("bm_sdp", 1, base + 3300)]
    row += [("br_acc", 0, 7000), ("br_epi", 0, 8200)]
    dec = tr.decode(buffer({"softmax0": row, "mma": mma, "tma": tma}), 1, 64)
    s = tr.summarize_bwd(dec)
    assert s["row.first.wait_for_S"]["median"] == 600 and s["row.steady.work_S_to_P"]["median"] == 1300
    assert s["stage.block_period"]["median"] == 3000
    assert s["handoff.row_P_to_mma_P"]["median"] == 100
    assert s["mma.issue_acc"]["median"] == 600
    assert sorted([s["mma.issue_S_dP"]["p10"], s["mma.issue_S_dP"]["p90"]]) == [390, 600]
    assert s["row.epilogue"]["median"] == 1200
    # S / dP issued at 400 and 3400, seen by the row warps at 700 and 3700
    assert s["handoff.S_dP_issue_to_row_S"]["median"] == 300 and s["handoff.S_dP_issue_to_row_S"]["n"] == 2
    # half-tiles: issued at 2, 3; the MMA found them ready at 10 and 2800
    assert s["tma.half_tile_issue_to_mma_ready"]["n"] == 2


def test_abi_rejects_bad_backward_trace_options_before_cuda():
    import exact_attention_forward_08_gb300 as fa
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    fa.load_library()
    fake = 0x10000
    args = (fake,) * 9 + (1, 2, 2, 128, 128)
    o = fa.default_options()
    o.trace, o.trace_ctas, o.trace_cap = fake, 0, 10
    assert fa.fa_bwd(*args, 128, 128, 0, 0.0, fake, 1 << 20, None, o) == fa.FA_ERR_INVALID_ARG
    o.trace_ctas = 1
    # the event-log build is made for head dims 128 only
    assert fa.fa_bwd(*args, 64, 64, 0, 0.0, fake, 1 << 20, None, o) == fa.FA_ERR_UNSUPPORTED
