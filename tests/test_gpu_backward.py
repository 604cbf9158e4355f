"""Backward pass on the GPU (through the C ABI) against the fp64 oracle.

The forward's O and LSE come from the CUDA forward; dO is seeded N(0,1) bf16.
The oracle differentiates the exact definition from the same bf16 inputs.
Head dims (64, 64), (128, 128) and (192, 128).
Tolerance, relative to the size of each reference gradient: the bf16 P, dS
and outputs carry 2^-9 (2e-3) relative rounding, and the measured errors on
these cases are 2-5e-3 of max|ref| at the worst element and 2.3e-3 of
mean|ref| on average.  Bounds: max|d - ref| <= 2e-2 * max(max|ref|, 1e-3)
and mean|d - ref| <= 1e-2 * max(mean|ref|, 1e-3) per gradient; the 1e-3
floor covers gradients that vanish exactly (one key: P = 1, so dS = 0 and
dQ = dK = 0, where the GPU leaves rounding of order 1e-7).  The wide-range
input (Q x 4, keys with a rising offset) has its own bounds (bounds()).
"""
import zlib

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 2e-2, 1e-2
WIDE_MAX_REL, WIDE_MEAN_REL = 5e-2, 3e-2  # the wide-range input (see bounds())


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run(fa, w, seed):
    q, k, v = w.generate()
    g = synthetic.normal_bf16(w.shapes["o"], seed, 7)
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    o, lse = fa.attention_forward(qd, kd, vd, causal=w.causal, scale=w.softmax_scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, gd, causal=w.causal, scale=w.softmax_scale)
    torch.cuda.synchronize()
    code, detail = fa.fa_device_status()
    assert code == 0, f"device status {code} {detail}"
    return (q, k, v, g), (dq, dk, dv)


def bounds(w):
    """(max, mean) relative bounds: the unit-normal ones, or the wide-range
    input's (Q x 4, keys with a rising offset).  There the softmax is nearly
    one-hot, so the dominant key's dS = P (dP - D) is a small difference of
    two terms that carry D's 2^-8 relative error (D from the bf16 O), and the
    large Q and K carry it into dQ and dK."""
    if w.q_mul == 1.0 and w.k_offset == 0.0:
        return MAX_REL, MEAN_REL
    return WIDE_MAX_REL, WIDE_MEAN_REL


def check(w, inputs, grads, what):
    q, k, v, g = inputs
    ref = oracle.attn_bwd(q, k, v, g, causal=w.causal, scale=w.softmax_scale)
    max_rel, mean_rel = bounds(w)
    out = {}
    for name, got, want in zip(("dq", "dk", "dv"), grads, ref):
        got = got.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"{what} {name}: non-finite"
        err = np.abs(got - want)
        scale_max = max(float(np.abs(want).max()), 1e-3)
        scale_mean = max(float(np.abs(want).mean()), 1e-3)
        out[name] = (float(err.max()) / scale_max, float(err.mean()) / scale_mean)
        print(f"{what} {name}: max {out[name][0]:.2e} mean {out[name][1]:.2e} (|ref| max {scale_max:.3g})")
        assert err.max() <= max_rel * scale_max, f"{what} {name}: max rel {out[name][0]:.3e}"
        assert err.mean() <= mean_rel * scale_mean, f"{what} {name}: mean rel {out[name][1]:.3e}"
    return out


CASES = [
    # name, B, Hq, Hkv, Sq, Sk, d, causal
    ("b_tiny", 1, 2, 2, 128, 128, 64, False),
    ("b_causal", 2, 4, 2, 300, 300, 128, True),
    ("b_sq_lt_sk", 1, 8, 2, 200, 456, 128, True),
    ("b_empty_rows", 1, 4, 2, 456, 200, 128, True),
    ("b_mqa", 1, 8, 1, 257, 257, 64, True),
    ("b_ragged", 2, 2, 2, 700, 530, 128, False),
    ("b_many", 2, 8, 8, 1300, 1300, 64, True),
    ("b_one_key", 1, 2, 1, 5, 1, 64, False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_small(fa, case):
    name, B, Hq, Hkv, Sq, Sk, d, causal = case
    w = synthetic.Workload(name, B, Hq, Hkv, Sq, Sk, d, d, causal, seed=zlib.crc32(name.encode()) % 1000)
    inputs, grads = run(fa, w, 11)
    check(w, inputs, grads, name)


ASYM_CASES = [
    # name, B, Hq, Hkv, Sq, Sk, causal, extra: head dims (d_qk, d_v) = (192, 128)
    ("ba_causal", 1, 4, 4, 300, 300, True, {}),
    ("ba_noncausal_ragged", 2, 2, 2, 257, 513, False, {}),
    ("ba_gqa", 1, 8, 2, 500, 500, True, {}),
    ("ba_empty_rows", 1, 4, 2, 456, 200, True, {}),
    ("ba_wide_range", 1, 4, 4, 640, 640, True, dict(q_mul=4.0, k_offset=12.0)),
    ("ba_wide_range_nc", 1, 4, 4, 640, 640, False, dict(q_mul=4.0, k_offset=12.0)),
    ("ba_many", 2, 4, 4, 1300, 1300, True, {}),
]


@pytest.mark.parametrize("case", ASYM_CASES, ids=[c[0] for c in ASYM_CASES])
def test_backward_asymmetric_head_dims(fa, case):
    """d_qk = 192, d_v = 128: the dK/dV kernel's S and dP share TMEM columns,
    the dQ kernel reads Q and dO from shared memory."""
    name, B, Hq, Hkv, Sq, Sk, causal, extra = case
    w = synthetic.Workload(name, B, Hq, Hkv, Sq, Sk, 192, 128, causal, seed=zlib.crc32(name.encode()) % 1000,
                           **extra)
    inputs, grads = run(fa, w, 12)
    assert grads[0].shape[-1] == 192 and grads[1].shape[-1] == 192 and grads[2].shape[-1] == 128
    check(w, inputs, grads, name)


def test_backward_wide_range_d128(fa):
    """The wide-range input at (128, 128): the same D-limited accuracy as at
    (192, 128), so it is a property of D from the bf16 O, not of the head dims."""
    w = synthetic.Workload("b_wide_range", 1, 4, 4, 640, 640, 128, 128, True, seed=361, q_mul=4.0, k_offset=12.0)
    inputs, grads = run(fa, w, 12)
    check(w, inputs, grads, "b_wide_range")


def test_backward_asymmetric_paired_and_deterministic(fa):
    """(192, 128), causal: the paired order over several grids is
    bit-identical to the plain order, and repeat runs are bit-identical."""
    w = synthetic.Workload("ba_pair", 1, 4, 4, 1024, 1024, 192, 128, True, seed=44)
    q, k, v = w.generate()
    g = synthetic.normal_bf16(w.shapes["o"], 13, 7)
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=w.softmax_scale)

    def grads(no_balance, grid):
        opts = fa.default_options()
        opts.no_balance = no_balance
        opts.grid = grid
        outs = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
        fa.attention_backward(qd, kd, vd, o, lse, gd, causal=True, scale=w.softmax_scale, dq=outs[0], dk=outs[1],
                              dv=outs[2], options=opts)
        torch.cuda.synchronize()
        code, detail = fa.fa_device_status()
        assert code == 0, f"device status {code} {detail}"
        return outs

    plain = grads(1, 0)
    for grid in (0, 5, 0):
        for a, b in zip(grads(0, grid), plain):
            assert torch.equal(a, b), grid
    check(w, (q, k, v, g), plain, "ba_pair")


def test_backward_deterministic(fa):
    w = synthetic.Workload("det", 2, 4, 2, 600, 600, 128, 128, True, seed=5)
    _, g1 = run(fa, w, 3)
    _, g2 = run(fa, w, 3)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_backward_degenerate(fa):
    q = torch.randn(1, 0, 2, 64, device="cuda").to(torch.bfloat16)
    k = torch.randn(1, 10, 2, 64, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 0, device="cuda")
    dq, dk, dv = fa.attention_backward(q, k, k, o, lse, o)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)


@pytest.mark.slow
@pytest.mark.parametrize("causal", [False, True])
def test_backward_mid_size_full(fa, causal):
    """Every element of dQ, dK, dV at a size spanning many tiles and both
    kernels' task orders (32 x 32 key x query blocks per head)."""
    w = synthetic.Workload("bmid", 1, 4, 2, 4096, 4096, 128, 128, causal, seed=21 + int(causal))
    inputs, grads = run(fa, w, 17)
    check(w, inputs, grads, f"mid causal={causal}")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["causal1k", "causal8k"])
def test_backward_benchmark_configs_full(fa, name):
    """Every element of dQ, dK, dV of two benchmark configurations at full
    size (the inputs and dO the backward bench uses), in the launch it times:
    the short causal tasks and the long paired ones."""
    w = synthetic.workloads()[name]
    inputs, grads = run(fa, w, w.seed)
    check(w, inputs, grads, f"full {name}")


# Paired causal order of the backward kernels: the task of heaviness rank q
# and its complement (blocks - 1 - q) on one CTA in consecutive waves.  Every
# task computes what it computes in the plain order, so the gradients (written
# over NaN, so a task left out would show) must be bit-identical to it.
PAIRED = [
    # name, B, Hq, Hkv, S, d, grids
    ("bp_even", 2, 4, 2, 1024, 128, (0, 5, 7)),      # 8 blocks
    ("bp_gqa", 1, 8, 2, 2048, 64, (0, 3, 11)),       # 16 blocks, 4 query heads per K/V head
    ("bp_odd_blocks", 1, 4, 4, 640, 128, (0, 3)),    # 5 blocks: plain order
    ("bp_sq_lt_sk", 1, 4, 4, 1000, 1500, 64, (0, 6)),
]


@pytest.mark.parametrize("case", PAIRED, ids=[c[0] for c in PAIRED])
def test_backward_paired_order_bitwise(fa, case):
    if len(case) == 8:
        name, B, Hq, Hkv, Sq, Sk, d, grids = case
    else:
        name, B, Hq, Hkv, Sq, d, grids = case
        Sk = Sq
    w = synthetic.Workload(name, B, Hq, Hkv, Sq, Sk, d, d, True, seed=zlib.crc32(name.encode()) % 1000)
    q, k, v = w.generate()
    g = synthetic.normal_bf16(w.shapes["o"], 13, 7)
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=w.softmax_scale)

    def grads(no_balance, grid):
        opts = fa.default_options()
        opts.no_balance = no_balance
        opts.grid = grid
        outs = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
        fa.attention_backward(qd, kd, vd, o, lse, gd, causal=True, scale=w.softmax_scale, dq=outs[0], dk=outs[1],
                              dv=outs[2], options=opts)
        torch.cuda.synchronize()
        code, detail = fa.fa_device_status()
        assert code == 0, f"device status {code} {detail}"
        return outs

    plain = grads(1, 0)
    for t in plain:
        assert torch.isfinite(t.float()).all()
    for grid in grids:
        for a, b in zip(grads(0, grid), plain):
            assert torch.equal(a, b), (name, grid)
    check(w, (q, k, v, g), plain, name)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_event_log_build(fa, causal):
    """The event-log build of both backward kernels (fa_options.trace, head
    dims 128): gradients bit-identical to the default build; with every CTA
    recording, each stage's row warps log one S wait and one P arrival per
    streamed block, as many as the MMA warp logs P waits, which is the task
    count times the blocks each task streams (non-causal: B Hq mq nk in both
    kernels)."""
    from exact_attention_forward_08_gb300 import trace as tr
    B, Hq, Hkv, S = 2, 4, 2, 640
    w = synthetic.Workload("b_trace", B, Hq, Hkv, S, S, 128, 128, causal, seed=77)
    q, k, v = w.generate()
    g = synthetic.normal_bf16(w.shapes["o"], 78, 7)
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=w.softmax_scale)
    ref = fa.attention_backward(qd, kd, vd, o, lse, gd, causal=causal, scale=w.softmax_scale)
    grid, cap = 3, 4096
    words = tr.trace_words(grid, cap)
    buf = torch.zeros(2 * words, dtype=torch.int64, device="cuda")
    opts = fa.default_options()
    opts.grid = grid
    opts.trace, opts.trace_ctas, opts.trace_cap = buf.data_ptr(), grid, cap
    got = fa.attention_backward(qd, kd, vd, o, lse, gd, causal=causal, scale=w.softmax_scale, options=opts)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == fa.FA_OK
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    host = buf.cpu().numpy().view(np.uint64)
    mq = nk = (S + 127) // 128
    for kind in (0, 1):
        ctas = tr.decode(host[kind * words:(kind + 1) * words], grid, cap)
        for s in (0, 1):
            p_row = sum(1 for c in ctas for _, ev, _ in c[f"softmax{s}"] if ev == "br_p")
            s_row = sum(1 for c in ctas for _, ev, _ in c[f"softmax{s}"] if ev == "br_s")
            p_mma = sum(1 for c in ctas for _, ev, arg in c["mma"] if ev == "bm_p" and arg >> 16 == s)
            assert p_row == s_row == p_mma, (kind, s, p_row, s_row, p_mma)
            if not causal:
                assert p_row == B * Hq * mq * nk, (kind, s, p_row)
        for c in ctas:
            for name in ("softmax0", "softmax1", "mma", "tma"):
                times = [t for t, _, _ in c[name]]
                assert times == sorted(times), name
        summ = tr.summarize_bwd(ctas)
        assert summ["row.steady.work_S_to_P"]["n"] > 0 and summ["mma.issue_acc"]["n"] > 0
    # head dims other than 128 are not built with the log
    w64 = synthetic.Workload("b_trace64", 1, 2, 2, 128, 128, 64, 64, False, seed=3)
    q6, k6, v6 = (to_dev(a) for a in w64.generate())
    o6, l6 = fa.attention_forward(q6, k6, v6)
    with pytest.raises(fa.FaError) as e:
        fa.attention_backward(q6, k6, v6, o6, l6, o6, options=opts)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
