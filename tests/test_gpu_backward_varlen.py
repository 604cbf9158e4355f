"""Backward of variable-length batches on the GPU (through the C ABI) against
the fp64 oracle: each sequence its own problem (oracle.attn_bwd_varlen,
pinned on the CPU to a packed brute-force backward).

Tolerances as the fixed-length backward tests: per gradient,
max|d - ref| <= 2e-2 max|ref| and mean|d - ref| <= 1e-2 mean|ref| (floors
1e-3), over the rows that lie in a sequence.  Also: equal lengths reproduce
the fixed-length backward bit for bit, rows outside every sequence are never
written, repeat runs are bitwise equal, bad offsets are reported on the device
with nothing computed, and the degenerate totals.
"""
import zlib

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 2e-2, 1e-2


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


def make(name, lq, lk, Hq, Hkv, d, dv, causal):
    return synthetic.VarlenWorkload(name, tuple(lq), tuple(lk), Hq, Hkv, d, dv, causal,
                                    seed=zlib.crc32(name.encode()) % 1000)


def grads(fa, w, q, k, v, g, **kw):
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    cq, ck = cu_dev(w.cu_seqlens_q), cu_dev(w.cu_seqlens_k)
    o, lse = fa.attention_forward_varlen(qd, kd, vd, cq, ck, causal=w.causal, scale=w.softmax_scale)
    out = fa.attention_backward_varlen(qd, kd, vd, o, lse, gd, cq, ck, causal=w.causal, scale=w.softmax_scale, **kw)
    torch.cuda.synchronize()
    code, detail = fa.fa_device_status()
    assert code == 0, f"device status {code} {detail}"
    return out


def inputs(w):
    q, k, v = w.generate()
    g = synthetic.normal_bf16((w.total_q, w.heads_q, w.d_v), w.seed, 7)
    return q, k, v, g


def check(w, q, k, v, g, got):
    ref = oracle.attn_bwd_varlen(q, k, v, g, w.cu_seqlens_q, w.cu_seqlens_k, causal=w.causal, scale=w.softmax_scale)
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        a = a.float().cpu().numpy().astype(np.float64)
        inside = np.isfinite(b)
        if not inside.any():
            continue
        assert np.all(np.isfinite(a[inside])), f"{w.name} {name}: non-finite"
        err = np.abs(a[inside] - b[inside])
        smax = max(float(np.abs(b[inside]).max()), 1e-3)
        smean = max(float(np.abs(b[inside]).mean()), 1e-3)
        print(f"{w.name} {name}: max {err.max() / smax:.2e} mean {err.mean() / smean:.2e}")
        assert err.max() <= MAX_REL * smax, f"{w.name} {name}: max rel {err.max() / smax:.3e}"
        assert err.mean() <= MEAN_REL * smean, f"{w.name} {name}: mean rel {err.mean() / smean:.3e}"


CASES = [
    # name, lengths q, lengths k, Hq, Hkv, d_qk, d_v, causal
    ("vb_mixed", (127, 0, 300, 1, 513, 128, 129), (127, 5, 300, 1, 513, 128, 129), 4, 2, 128, 128, True),
    ("vb_mixed_nc", (127, 0, 300, 1, 513, 128, 129), (127, 5, 300, 1, 513, 128, 129), 4, 2, 128, 128, False),
    ("vb_sq_ne_sk", (200, 456, 64), (456, 200, 0), 8, 2, 128, 128, True),
    ("vb_gqa4_d64", (300, 77, 640), (300, 77, 640), 8, 2, 64, 64, True),
    ("vb_mqa", (257, 33), (257, 33), 8, 1, 64, 64, False),
    ("vb_asym", (400, 129, 700), (400, 129, 700), 4, 4, 192, 128, True),
    ("vb_many", tuple(int(x) for x in np.random.default_rng(7).integers(1, 400, 30)),
     tuple(int(x) for x in np.random.default_rng(8).integers(1, 400, 30)), 4, 2, 128, 128, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_varlen_against_oracle(fa, case):
    w = make(*case)
    q, k, v, g = inputs(w)
    check(w, q, k, v, g, grads(fa, w, q, k, v, g))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_equal_lengths_match_fixed_length_bitwise(fa, causal, d):
    B, S, Hq, Hkv = 3, 384, 4, 2
    w = make(f"vb_eq_{d}_{int(causal)}", (S,) * B, (S,) * B, Hq, Hkv, d, d, causal)
    q, k, v, g = inputs(w)
    got = grads(fa, w, q, k, v, g)
    qd, kd, vd, gd = (to_dev(a).view(B, S, -1, a.shape[-1]) for a in (q, k, v, g))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=w.softmax_scale)
    ref = fa.attention_backward(qd, kd, vd, o, lse, gd, causal=causal, scale=w.softmax_scale)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b.reshape(a.shape))


def test_rows_outside_sequences_untouched_and_repeatable(fa):
    w = make("vb_gaps", (100, 250), (130, 90), 4, 2, 128, 128, True)
    q, k, v, g = inputs(w)
    # packed tensors with 40 extra rows past the last sequence
    pad = lambda a: np.concatenate([a, np.zeros((40,) + a.shape[1:], dtype=a.dtype)])
    qd, kd, vd, gd = (to_dev(pad(a)) for a in (q, k, v, g))
    cq, ck = cu_dev(w.cu_seqlens_q), cu_dev(w.cu_seqlens_k)
    o, lse = fa.attention_forward_varlen(qd, kd, vd, cq, ck, causal=True, scale=w.softmax_scale)
    outs = []
    for _ in range(2):
        dq = torch.full_like(qd, float("nan"))
        dk = torch.full_like(kd, float("nan"))
        dv = torch.full_like(vd, float("nan"))
        fa.attention_backward_varlen(qd, kd, vd, o, lse, gd, cq, ck, causal=True, scale=w.softmax_scale,
                                     dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
        assert fa.fa_device_status()[0] == fa.FA_OK
        assert torch.isnan(dq[w.total_q:].float()).all() and torch.isnan(dk[w.total_k:].float()).all()
        assert torch.isnan(dv[w.total_k:].float()).all()
        outs.append((dq[:w.total_q].clone(), dk[:w.total_k].clone(), dv[:w.total_k].clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    check(w, q, k, v, g, outs[0])


def test_bad_offsets_reported(fa):
    w = make("vb_bad", (64, 64), (64, 64), 2, 2, 64, 64, False)
    q, k, v, g = inputs(w)
    qd, kd, vd, gd = (to_dev(a) for a in (q, k, v, g))
    cq = cu_dev(w.cu_seqlens_q)
    o, lse = fa.attention_forward_varlen(qd, kd, vd, cq, cu_dev(w.cu_seqlens_k))
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == fa.FA_OK
    bad_k = cu_dev([0, 100, 64])  # out of order
    dq = torch.full_like(qd, 7.0)
    fa.attention_backward_varlen(qd, kd, vd, o, lse, gd, cq, bad_k, dq=dq)
    torch.cuda.synchronize()
    code, detail = fa.fa_device_status()
    assert code == fa.FA_ERR_INVALID_ARG and detail[1] == 501 and detail[2] == 1, (code, detail)
    assert torch.all(dq == 7.0)  # nothing computed


def test_degenerate_totals(fa):
    k = torch.randn(10, 2, 64, device="cuda").to(torch.bfloat16)
    q = torch.empty(0, 2, 64, device="cuda", dtype=torch.bfloat16)
    o = torch.empty(0, 2, 64, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(2, 0, device="cuda")
    cq, ck = cu_dev([0, 0, 0]), cu_dev([0, 4, 10])
    dq, dk, dv = fa.attention_backward_varlen(q, k, k, o, lse, o, cq, ck)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
