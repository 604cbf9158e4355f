"""The forward kernel's debug builds, through the C ABI.

Checking build (fa_options.debug_flags bit 2): on the small parity problems,
with both epilogues, every range check and every hand-off count comparison
passes (status FA_OK), the output is bit-identical to the default kernel's,
and it matches the fp64 oracle.  A fault planted for the checks (debug bit 3:
task 0 decodes to an out-of-range batch index) is reported as
FA_ERR_DEVICE_CHECK at the task-check site before any access is made, and the
context computes correctly afterwards.

Event-log build (fa_options.trace): the output is bit-identical to the
default kernel's, and the log holds, for each recording CTA, as many S waits
and P arrivals per stage as the host plan gives K/V blocks to that CTA's
tiles, in increasing clock order.

Staggered-exponential ablation (fa_options.stagger): bit-identical output.

O-rescale counter (debug bit 1) in the checking build, whose arithmetic is the
default kernel's: on causal problems (the same task decomposition in every
build) it counts exactly what the FMA-exp2 ablation kernel counts, since the
rescale decisions depend only on the scores' row maxima, not on how the
exponentials are taken; and it counts rescales on the wide-range input.
"""
import zlib

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL = [
    # name, B, Hq, Hkv, Sq, Sk, dq, dv, causal, extra
    ("tiny", 1, 1, 1, 128, 128, 64, 64, False, {}),
    ("ragged", 2, 4, 4, 300, 300, 128, 128, False, {}),
    ("causal384", 2, 4, 4, 384, 384, 128, 128, True, {}),
    ("causal_sq_lt_sk", 1, 8, 2, 200, 456, 128, 128, True, {}),
    ("causal_empty_rows", 1, 8, 2, 456, 200, 128, 128, True, {}),
    ("gqa4", 1, 32, 8, 500, 500, 128, 128, True, {}),
    ("mqa32", 1, 32, 1, 300, 300, 128, 128, True, {}),
    ("ratio3", 1, 6, 2, 77, 77, 192, 128, True, {}),
    ("ratio256", 1, 256, 1, 20, 40, 64, 64, False, {}),
    ("asym_offset", 1, 16, 16, 1000, 1000, 192, 128, True, dict(q_mul=4.0, k_offset=12.0)),
    ("d64", 2, 4, 2, 257, 513, 64, 64, False, {}),
    ("d128_v64", 1, 3, 1, 140, 260, 128, 64, True, {}),
    ("d192_v64", 1, 3, 1, 40, 40, 192, 64, False, {}),
    ("one_key", 1, 2, 2, 1, 1, 128, 128, False, {}),
    ("short_k", 1, 2, 1, 5, 130, 128, 64, True, {}),
    ("sk_below_tile", 2, 2, 2, 70, 33, 64, 64, False, {}),
    ("many_tasks", 3, 8, 8, 1300, 1300, 64, 64, True, {}),
    # key-split last wave and paired causal order on a small grid
    ("tail_split", 1, 4, 4, 2048, 2048, 128, 128, False, dict(grid=5)),
    ("paired", 2, 4, 4, 1024, 1024, 128, 128, True, dict(grid=6)),
]


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def workload(case):
    name, B, Hq, Hkv, Sq, Sk, dq, dv, causal, extra = case
    extra = {k: v for k, v in extra.items() if k != "grid"}
    return synthetic.Workload(name, B, Hq, Hkv, Sq, Sk, dq, dv, causal, seed=zlib.crc32(name.encode()) % 1000,
                              **extra)


def options(fa, case, store_mode, flags=0):
    o = fa.default_options()
    o.store_mode = store_mode
    o.debug_flags = flags
    o.grid = case[9].get("grid", 0)
    return o


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_checking_build_passes_and_matches(fa, case):
    w = workload(case)
    qh, kh, vh = w.generate()
    q, k, v = to_dev(qh), to_dev(kh), to_dev(vh)
    assert fa.fa_device_status()[0] == fa.FA_OK
    for store_mode in (1, 2):
        ref = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale,
                                   options=options(fa, case, store_mode))
        got = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale,
                                   options=options(fa, case, store_mode, fa.DEBUG_CHECKS))
        torch.cuda.synchronize()
        code, detail = fa.fa_device_status()
        assert code == fa.FA_OK, (store_mode, detail)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), store_mode
    # and against the oracle (the default kernel's parity is tested elsewhere;
    # here the checking build's own output)
    o_ref, lse_ref = oracle.attn_fwd(qh, kh, vh, causal=w.causal, scale=w.softmax_scale)
    og = got[0].float().cpu().numpy().astype(np.float64)
    err = np.abs(og - o_ref)
    # the stated bound for unit-normal inputs; the arithmetic's 2^-7 max|V| for the wide-range input
    max_bound = 2e-2
    if w.q_mul != 1.0 or w.k_offset != 0.0:
        max_bound = 2.0 ** -7 * float(np.abs(synthetic.bf16_bits_to_f32(vh)).max())
    assert err.max() <= max_bound and err.mean() <= 2e-3
    lg = got[1].cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    if fin.any():
        assert np.abs(lg[fin] - lse_ref[fin]).max() <= 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_checking_build_catches_planted_fault(fa, causal):
    w = synthetic.Workload("plant", 2, 4, 4, 300, 300, 128, 128, causal, seed=5)
    qh, kh, vh = w.generate()
    q, k, v = to_dev(qh), to_dev(kh), to_dev(vh)
    assert fa.fa_device_status()[0] == fa.FA_OK
    opts = fa.default_options()
    opts.debug_flags = fa.DEBUG_CHECKS | fa.DEBUG_PLANT_BAD_TASK
    opts.timeout_s = 0.5
    fa.attention_forward(q, k, v, causal=causal, options=opts)
    code, detail = fa.fa_device_status()
    assert code == fa.FA_ERR_DEVICE_CHECK, (code, detail)
    assert detail[0] == 5 and detail[1] == 701, detail
    assert fa.fa_device_status()[0] == fa.FA_OK
    # the context still computes correctly
    o, lse = fa.attention_forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == fa.FA_OK
    o_ref, _ = oracle.attn_fwd(qh, kh, vh, causal=causal)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= 2e-2


def test_debug_builds_reject_unsupported_calls(fa):
    w = synthetic.Workload("rej", 1, 2, 2, 256, 256, 64, 64, False, seed=3)
    q, k, v = (to_dev(a) for a in w.generate())
    buf = torch.zeros(1 << 16, dtype=torch.int64, device="cuda")
    opts = fa.default_options()
    opts.trace, opts.trace_ctas, opts.trace_cap = buf.data_ptr(), 1, 100
    with pytest.raises(fa.FaError) as e:  # the event log is built for (128,128) and (192,128) only
        fa.attention_forward(q, k, v, options=opts)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    w = synthetic.Workload("rej", 1, 2, 2, 256, 256, 128, 128, False, seed=3)
    q, k, v = (to_dev(a) for a in w.generate())
    opts.debug_flags = fa.DEBUG_CHECKS  # one debug build at a time
    with pytest.raises(fa.FaError) as e:
        fa.attention_forward(q, k, v, options=opts)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    opts.debug_flags = 0
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:  # not with dynamic assignment
        fa.attention_forward(q, k, v, options=opts, workspace=ws)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    opts.trace_ctas = 0
    with pytest.raises(fa.FaError) as e:
        fa.attention_forward(q, k, v, options=opts)
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == fa.FA_OK


TRACE_CASES = [
    ("mha", 2, 8, 8, 1024, 1024, 128, 128, False, {}),
    ("causal", 2, 8, 8, 1024, 1024, 128, 128, True, {}),
    ("asym", 1, 4, 4, 1000, 1000, 192, 128, True, dict(q_mul=4.0, k_offset=12.0)),
    ("tail_split", 1, 4, 4, 2048, 2048, 128, 128, False, dict(grid=5)),
]


@pytest.mark.parametrize("case", TRACE_CASES, ids=[c[0] for c in TRACE_CASES])
@pytest.mark.parametrize("store_mode", [1, 2])
def test_event_log_build(fa, case, store_mode):
    from exact_attention_forward_08_gb300 import trace as tr
    w = workload(case)
    q, k, v = (to_dev(a) for a in w.generate())
    grid = case[9].get("grid", 0) or torch.cuda.get_device_properties(0).multi_processor_count
    ctas, cap = min(grid, 4), 4096
    buf = torch.zeros(tr.trace_words(ctas, cap), dtype=torch.int64, device="cuda")
    base = options(fa, case, store_mode)
    topts = options(fa, case, store_mode)
    topts.trace, topts.trace_ctas, topts.trace_cap = buf.data_ptr(), ctas, cap
    ref = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=base)
    got = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=topts)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == fa.FA_OK
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    dec = tr.decode(buf.cpu().numpy().view(np.uint64), ctas, cap)
    # the tasks each recording CTA ran, from the host copy of the schedule
    plan = fa.fa_make_plan(w.batch, w.heads_q, w.heads_kv, w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, int(w.causal))
    fa.fa_plan_set_grid(plan, grid)
    for c, cta in enumerate(dec):
        blocks = [0, 0]
        for t in range(c, plan.num_tasks, grid):
            task = fa.fa_plan_task(plan, t)
            for s in range(2):
                blocks[s] += task.n_blocks[s]
        for s in range(2):
            evs = cta[f"softmax{s}"]
            assert cta["_counts"][f"softmax{s}"] <= cap
            n_s = sum(1 for _, e, _ in evs if e == "sm_s")
            n_p = sum(1 for _, e, _ in evs if e == "sm_p")
            assert n_s == blocks[s] and n_p == blocks[s], (c, s, n_s, n_p, blocks)
            times = [t for t, _, _ in evs]
            assert times == sorted(times)
        mm = cta["mma"]
        assert sum(1 for _, e, _ in mm if e == "mm_pv") == blocks[0] + blocks[1]
        assert [t for t, _, _ in mm] == sorted(t for t, _, _ in mm)
    summary = tr.summarize(dec)
    assert summary["softmax.steady.work_S_to_P"]["median"] > 0
    assert summary["mma.issue_PV"]["median"] > 0


STAGGER_CASES = [c for c in SMALL if (c[6], c[7]) in ((128, 128), (192, 128))]


@pytest.mark.parametrize("case", STAGGER_CASES, ids=[c[0] for c in STAGGER_CASES])
def test_stagger_build_bitwise_equal(fa, case):
    """The staggered-exponential ablation changes only when each stage's
    exponentials run, not what they compute."""
    w = workload(case)
    q, k, v = (to_dev(a) for a in w.generate())
    for store_mode in (1, 2):
        base = options(fa, case, store_mode)
        st = options(fa, case, store_mode)
        st.stagger = 1
        ref = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=base)
        got = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=st)
        torch.cuda.synchronize()
        code, detail = fa.fa_device_status()
        assert code == fa.FA_OK, detail
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), store_mode


RESCALE_CASES = [c for c in SMALL if c[0] in ("causal384", "gqa4", "asym_offset", "many_tasks")]


@pytest.mark.parametrize("case", RESCALE_CASES, ids=[c[0] for c in RESCALE_CASES])
def test_rescale_counter_in_checking_build(fa, case):
    w = workload(case)
    q, k, v = (to_dev(a) for a in w.generate())
    assert fa.fa_device_status()[0] == fa.FA_OK
    counts = []
    for flags, emu in ((fa.DEBUG_CHECKS | fa.DEBUG_COUNT_RESCALE, 0), (fa.DEBUG_COUNT_RESCALE, 1)):
        opts = fa.default_options()
        opts.debug_flags, opts.exp_emu = flags, emu
        fa.fa_debug_rescale_count()  # clear
        fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=opts)
        counts.append(fa.fa_debug_rescale_count())
        assert fa.fa_device_status()[0] == fa.FA_OK
    assert counts[0] == counts[1], counts
    if case[0] == "asym_offset":
        assert counts[0] > 0
    # without either build the counter is refused
    opts = fa.default_options()
    opts.debug_flags = fa.DEBUG_COUNT_RESCALE
    with pytest.raises(fa.FaError) as e:
        fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=opts)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
