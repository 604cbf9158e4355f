"""Split-KV forward (decode / short-Q) on the GPU against the fp64 oracle.

The keys of every task are cut into ranges, each range's partial result goes
to the workspace, and the merge kernel combines them; the result is the same
attention, so it is compared with the oracle's definition at the usual
tolerances (max|dO| <= 2e-2, mean <= 2e-3, |dLSE| <= 1e-3, empty rows exactly
O = 0 and LSE = -inf)."""
import zlib

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def compare(og, lg, orf, lrf, what):
    empty = ~np.isfinite(lrf)
    assert np.array_equal(~np.isfinite(lg), empty), f"{what}: empty-row pattern differs"
    if empty.any():
        assert np.all(lg[empty] == -np.inf) and np.all(og[empty] == 0.0), f"{what}: empty rows"
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    err = np.abs(og - orf)
    lerr = float(np.abs(lg[~empty] - lrf[~empty]).max()) if (~empty).any() else 0.0
    assert err.max() <= 2e-2, f"{what}: max|dO| {err.max():.3e}"
    assert err.mean() <= 2e-3, f"{what}: mean|dO| {err.mean():.3e}"
    assert lerr <= 1e-3, f"{what}: max|dLSE| {lerr:.3e}"


def run_split(fa, w, q, k, v, splits):
    o, lse = fa.attention_forward_splitkv(to_dev(q), to_dev(k), to_dev(v), causal=w.causal, scale=w.softmax_scale,
                                          num_splits=splits)
    torch.cuda.synchronize()
    code, detail = fa.fa_device_status()
    assert code == 0, f"device status {code} {detail}"
    return o, lse


CASES = [
    # name, B, Hq, Hkv, Sq, Sk, dq, dv, causal
    ("dec_gqa4", 3, 8, 2, 1, 1000, 128, 128, False),
    ("dec_mqa", 2, 32, 1, 1, 4113, 128, 128, False),
    ("dec_mha_d64", 2, 4, 4, 1, 2600, 64, 64, False),
    ("dec_d192", 2, 6, 2, 1, 1500, 192, 128, False),
    ("spec4_causal", 4, 8, 8, 4, 3000, 64, 64, True),
    ("few_blocks", 1, 2, 1, 5, 130, 128, 64, True),
    ("prefill_causal", 1, 4, 4, 700, 700, 128, 128, True),
    ("empty_rows", 1, 4, 2, 456, 200, 128, 128, True),
]


@pytest.mark.parametrize("splits", [0, 1, 2, 3, 7, 64])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_splitkv_full(fa, case, splits):
    name, B, Hq, Hkv, Sq, Sk, dq, dv, causal = case
    w = synthetic.Workload(name, B, Hq, Hkv, Sq, Sk, dq, dv, causal, seed=zlib.crc32(name.encode()) % 1000)
    q, k, v = w.generate()
    o, lse = run_split(fa, w, q, k, v, splits)
    orf, lrf = oracle.attn_fwd(q, k, v, causal=causal, scale=w.softmax_scale)
    og = o.float().cpu().numpy().astype(np.float64).reshape(-1, dv)
    lg = lse.cpu().numpy().astype(np.float64).transpose(0, 2, 1).reshape(-1)
    compare(og, lg, orf.reshape(-1, dv), lrf.transpose(0, 2, 1).reshape(-1), f"{name} splits={splits}")


def test_one_split_is_the_plain_kernel_bitwise(fa):
    w = synthetic.Workload("one", 2, 8, 2, 3, 900, 128, 128, True, seed=3)
    q, k, v = (to_dev(a) for a in w.generate())
    o1, l1 = fa.attention_forward(q, k, v, causal=True)
    o2, l2 = fa.attention_forward_splitkv(q, k, v, causal=True, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_repeat_bit_identical_and_workspace_reuse(fa):
    w = synthetic.Workload("rep", 4, 16, 4, 1, 5000, 128, 128, False, seed=4)
    q, k, v = (to_dev(a) for a in w.generate())
    ws = torch.full((fa.fa_splitkv_workspace_size(4, 16, 1, 128, 9),), 0x55, dtype=torch.uint8, device="cuda")
    o1, l1 = fa.attention_forward_splitkv(q, k, v, num_splits=9, workspace=ws)
    o2, l2 = fa.attention_forward_splitkv(q, k, v, num_splits=9, workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode32k", "decode_mqa", "specdec"])
def test_decode_workloads_full(fa, name):
    w = synthetic.decode_workloads()[name]
    q, k, v = w.generate()
    o, lse = run_split(fa, w, q, k, v, 0)
    orf, lrf = oracle.attn_fwd(q, k, v, causal=w.causal, scale=w.softmax_scale)
    og = o.float().cpu().numpy().astype(np.float64).reshape(-1, w.d_v)
    lg = lse.cpu().numpy().astype(np.float64).transpose(0, 2, 1).reshape(-1)
    compare(og, lg, orf.reshape(-1, w.d_v), lrf.transpose(0, 2, 1).reshape(-1), name)
