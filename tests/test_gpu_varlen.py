"""Variable-length batches on the GPU through the C ABI, against the fp64
oracle (each sequence its own attention problem).

Same tolerances as the fixed-length parity tests: max|dO| <= 2e-2,
mean|dO| <= 2e-3, |dLSE| <= 1e-3, rows with no visible key exactly O = 0 and
LSE = -inf.  Also: the planning kernel writes exactly the host plan, rows
outside every sequence are never written, equal lengths reproduce the
fixed-length kernel bit for bit, and bad offsets are reported on the device.
"""
import zlib

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_TOL, MEAN_TOL, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def cu_dev(cu):
    return torch.tensor(np.asarray(cu, dtype=np.int32), device="cuda")


def status(fa):
    torch.cuda.synchronize()
    return fa.fa_device_status()


def compare(og, lg, orf, lrf, what):
    empty = ~np.isfinite(lrf)
    assert np.array_equal(~np.isfinite(lg), empty), f"{what}: empty-row pattern differs"
    if empty.any():
        assert np.all(lg[empty] == -np.inf) and np.all(og[empty] == 0.0), f"{what}: empty rows"
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    err = np.abs(og - orf)
    lerr = float(np.abs(lg[~empty] - lrf[~empty]).max()) if (~empty).any() else 0.0
    assert err.max() <= MAX_TOL, f"{what}: max|dO| {err.max():.3e}"
    assert err.mean() <= MEAN_TOL, f"{what}: mean|dO| {err.mean():.3e}"
    assert lerr <= LSE_TOL, f"{what}: max|dLSE| {lerr:.3e}"


def make(name, lq, lk, Hq, Hkv, dq, dv, causal):
    return synthetic.VarlenWorkload(name, tuple(lq), tuple(lk), Hq, Hkv, dq, dv, causal,
                                    seed=zlib.crc32(name.encode()) % 1000)


def run(fa, w, q, k, v, **kw):
    o, lse = fa.attention_forward_varlen(to_dev(q), to_dev(k), to_dev(v), cu_dev(w.cu_seqlens_q),
                                         cu_dev(w.cu_seqlens_k), causal=w.causal, scale=w.softmax_scale, **kw)
    code, detail = status(fa)
    assert code == 0, f"device status {code} {detail}"
    return o, lse


def full_check(fa, w):
    q, k, v = w.generate()
    o, lse = run(fa, w, q, k, v)
    orf, lrf = oracle.attn_fwd_varlen(q, k, v, w.cu_seqlens_q, w.cu_seqlens_k, causal=w.causal,
                                      scale=w.softmax_scale)
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    compare(og.reshape(-1, w.d_v), lg.T.reshape(-1), orf.reshape(-1, w.d_v), lrf.T.reshape(-1), w.name)


EDGE = (1, 127, 128, 129, 0, 300, 513, 64)
rng = np.random.default_rng(2024)
MANY = tuple(int(x) for x in rng.integers(0, 400, 40))

SMALL = [
    ("v_causal", EDGE, EDGE, 4, 2, 128, 128, True),
    ("v_noncausal", EDGE, EDGE, 4, 2, 128, 128, False),
    ("v_sq_ne_sk", (200, 456, 5, 130), (456, 200, 130, 5), 8, 2, 128, 128, True),
    ("v_gqa_pack4", (300, 77, 513), (300, 77, 513), 32, 8, 128, 128, True),
    ("v_mqa", (257, 1, 129), (257, 1, 129), 32, 1, 128, 128, True),
    ("v_ratio3", (77, 200), (90, 200), 6, 2, 192, 128, True),
    ("v_d64", (257, 40, 0, 513), (513, 40, 9, 257), 4, 2, 64, 64, False),
    ("v_d128_v64", (140, 3), (260, 300), 3, 1, 128, 64, True),
    ("v_d192_v64", (40, 41), (40, 41), 3, 1, 192, 64, False),
    ("v_zero_keys", (50, 70, 10), (0, 90, 0), 4, 4, 128, 128, True),
    ("v_many", MANY, MANY, 4, 4, 64, 64, True),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_varlen_small_full(fa, case):
    full_check(fa, make(*case))


def test_device_plan_equals_host_plan(fa):
    w = make("plan", (300, 1, 0, 513, 129, 700), (400, 1, 5, 513, 0, 350), 8, 2, 128, 128, True)
    q, k, v = w.generate()
    ws = torch.zeros(fa.fa_varlen_workspace_size(w.batch, w.heads_q, w.total_q), dtype=torch.uint8, device="cuda")
    run(fa, w, q, k, v, workspace=ws)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size // 2
    host = fa.fa_varlen_plan_host(w.cu_seqlens_q, w.cu_seqlens_k, w.heads_q, w.heads_kv, w.d_qk, w.d_v, w.causal,
                                  l2_bytes=l2)
    raw = ws.cpu().numpy()
    count = int(raw[:4].view(np.int32)[0])
    assert count == len(host)
    recs = raw[fa.VARLEN_HEADER_BYTES:fa.VARLEN_HEADER_BYTES + 32 * count].view(np.int32).reshape(count, 8)
    want = np.array([[r.b, r.g, r.mblock, r.reserved, r.q_row0, r.seqlen_q, r.k_row0, r.seqlen_k] for r in host])
    assert np.array_equal(recs, want)


def test_rows_outside_sequences_untouched(fa):
    Hq, d = 4, 128
    total_q, total_k = 700, 600
    cu_q, cu_k = [3, 200, 650], [10, 300, 590]  # rows 0..2 and 650..699 of q / o belong to no sequence
    q = synthetic.normal_bf16((total_q, Hq, d), 7, 1)
    k = synthetic.normal_bf16((total_k, Hq, d), 7, 2)
    v = synthetic.normal_bf16((total_k, Hq, d), 7, 3)
    o = torch.full((total_q, Hq, d), 5.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((Hq, total_q), 9.0, dtype=torch.float32, device="cuda")
    for causal in (False, True):
        fa.attention_forward_varlen(to_dev(q), to_dev(k), to_dev(v), cu_dev(cu_q), cu_dev(cu_k), causal=causal,
                                    out=o, lse=lse)
        assert status(fa)[0] == 0
        og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
        assert np.all(og[:3] == 5.0) and np.all(og[650:] == 5.0)
        assert np.all(lg[:, :3] == 9.0) and np.all(lg[:, 650:] == 9.0)
        orf, lrf = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, causal=causal)
        compare(og[3:650].reshape(-1, d).astype(np.float64), lg[:, 3:650].T.reshape(-1).astype(np.float64),
                orf[3:650].reshape(-1, d), lrf[:, 3:650].T.reshape(-1), f"gaps causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_fixed_length_kernel_bitwise(fa, causal):
    B, S, Hq, Hkv, d = 3, 700, 8, 2, 128
    w = synthetic.Workload("eq", B, Hq, Hkv, S, S, d, d, causal, seed=77)
    q, k, v = w.generate()
    whole = fa.default_options()
    whole.no_balance = 1  # the varlen kernel runs whole tasks
    o_f, l_f = fa.attention_forward(to_dev(q), to_dev(k), to_dev(v), causal=causal, options=whole)
    cu = np.arange(B + 1) * S
    o_v, l_v = fa.attention_forward_varlen(to_dev(q.reshape(B * S, Hq, d)), to_dev(k.reshape(B * S, Hkv, d)),
                                           to_dev(v.reshape(B * S, Hkv, d)), cu_dev(cu), cu_dev(cu), causal=causal)
    assert status(fa)[0] == 0
    assert torch.equal(o_v.view(B, S, Hq, d), o_f)
    assert torch.equal(l_v.view(Hq, B, S).permute(1, 0, 2), l_f)


def test_bad_offsets_reported_on_device(fa):
    Hq, d = 2, 64
    q = to_dev(synthetic.normal_bf16((100, Hq, d), 1, 1))
    k = to_dev(synthetic.normal_bf16((100, Hq, d), 1, 2))
    o = torch.full((100, Hq, d), 3.0, dtype=torch.bfloat16, device="cuda")
    status(fa)
    for cu_q, cu_k, bad in (([0, 50, 40], [0, 50, 100], 1), ([0, 50, 101], [0, 50, 100], 1),
                            ([0, 50, 100], [-1, 50, 100], 0)):
        fa.attention_forward_varlen(q, k, k, cu_dev(cu_q), cu_dev(cu_k), out=o)
        code, detail = status(fa)
        assert code == fa.FA_ERR_INVALID_ARG and detail[1] == 501 and detail[2] == bad, (cu_q, cu_k, detail)
        assert torch.all(o == 3.0)
    # the context is still usable
    fa.attention_forward_varlen(q, k, k, cu_dev([0, 50, 100]), cu_dev([0, 50, 100]), out=o)
    assert status(fa)[0] == 0 and torch.all(torch.isfinite(o.float()))


def test_no_keys_anywhere(fa):
    Hq, d = 4, 128
    q = to_dev(synthetic.normal_bf16((90, Hq, d), 2, 1))
    k = torch.empty((0, Hq, d), dtype=torch.bfloat16, device="cuda")
    o, lse = fa.attention_forward_varlen(q, k, k, cu_dev([0, 40, 90]), cu_dev([0, 0, 0]), causal=True)
    assert status(fa)[0] == 0
    assert torch.all(o == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)


def test_repeat_runs_bit_identical(fa):
    w = make("det", (900, 300, 1200), (900, 300, 1200), 8, 8, 128, 128, True)
    q, k, v = w.generate()
    o1, l1 = run(fa, w, q, k, v)
    o2, l2 = run(fa, w, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["varlen32k", "varlen32k_nc"])
def test_varlen_full_size_sampled(fa, name):
    w = synthetic.varlen_workloads()[name]
    q, k, v = w.generate()
    o, lse = run(fa, w, q, k, v)
    cu = w.cu_seqlens_q
    r = np.random.default_rng(zlib.crc32(name.encode()))
    picks = []
    for b in range(w.batch):  # first and last row of every sequence, and random rows
        for t in (cu[b], cu[b + 1] - 1, *r.integers(cu[b], cu[b + 1], 2)):
            picks.append((int(t), int(r.integers(0, w.heads_q))))
    rows = np.array(picks)
    orf, lrf = oracle.attn_fwd_varlen(q, k, v, cu, w.cu_seqlens_k, causal=w.causal, scale=w.softmax_scale,
                                      rows=rows)
    og = o.float().cpu().numpy().astype(np.float64)[rows[:, 0], rows[:, 1]]
    lg = lse.cpu().numpy().astype(np.float64)[rows[:, 1], rows[:, 0]]
    compare(og, lg, orf, lrf, name)
