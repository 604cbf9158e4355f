"""Pins for the fp64 oracle: what the pages and the mathematics fix.

Each ``check_*`` takes an ``attn`` callable with the signature of
``oracle.attn_fwd`` so that ``test_pins_catch_planted_mistakes`` can run the
same checks against copies of the oracle with a mistake planted in them.

Pinned facts:
* the worked example of "Infra: Flash Attention", section "How softmax is
  computed in pieces" (exponentials 1, 2, 4, 8; values 1..4; O = 49/15),
  including the intermediate block states of its merge figure;
* closed forms: uniform scores give the mean of V and L = log(#keys); causal
  row 0 gives V_0 and L = scale q_0.k_0;
* invariants: softmax rows sum to one and have ratios e^{s_ij - s_ik}; key
  permutation equivariance; a constant key shift leaves O unchanged and moves
  L by scale q.w; GQA equals MHA on repeated K/V;
* brute force: pure-Python loops on tiny inputs, the bottom-right mask as a
  truncated non-causal problem;
* a library routine: torch float64 scaled_dot_product_attention plus
  logsumexp (the cross-check "Flash Attention 4 on Blackwell" uses in its
  "Build and validation constraints" section);
* the blocked and conditionally rescaled scans of ``oracle.online`` reach the
  definition for tau in {0, 8, inf}.
"""
import json
import math
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import online
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------
# checks (each raises AssertionError on failure)
# ----------------------------------------------------------------------------

def check_worked_example(attn):
    """O = 49/15 and L = log 15 for scores log(1,2,4,8), values 1..4, scale 1."""
    g = json.load(open(os.path.join(GOLDEN, "online_merge_49_15.json")))
    e = np.array(g["exp_scores"], dtype=np.float64)
    q = np.ones((1, 1, 1, 1))
    k = np.log(e).reshape(1, 4, 1, 1)
    v = np.array(g["values"], dtype=np.float64).reshape(1, 4, 1, 1)
    o, lse = attn(q, k, v, causal=False, scale=1.0)
    want = g["output"]["numerator"] / g["output"]["denominator"]
    assert abs(o[0, 0, 0, 0] - want) < 1e-13, (o, want)
    assert abs(lse[0, 0, 0] - math.log(e.sum())) < 1e-13


def check_uniform_scores(attn):
    """q = 0: every visible key has the same score, O = mean of visible V, L = log count."""
    r = _rng(1)
    B, Sq, Sk, Hq, Hkv, d, dv = 2, 5, 7, 4, 2, 8, 3
    q = np.zeros((B, Sq, Hq, d))
    k = r.normal(size=(B, Sk, Hkv, d))
    v = r.normal(size=(B, Sk, Hkv, dv))
    for causal in (False, True):
        o, lse = attn(q, k, v, causal=causal, scale=0.37)
        for b in range(B):
            for i in range(Sq):
                n = Sk if not causal else min(Sk, i + Sk - Sq + 1)
                for h in range(Hq):
                    kv = h // (Hq // Hkv)
                    np.testing.assert_allclose(o[b, i, h], v[b, :n, kv].mean(axis=0), rtol=0, atol=1e-13)
                    assert abs(lse[b, h, i] - math.log(n)) < 1e-13


def check_probabilities(attn):
    """With V = identity (dv = Sk) the output row is the probability row itself."""
    r = _rng(2)
    Sq, Sk, d = 6, 9, 5
    q = r.normal(size=(1, Sq, 1, d))
    k = r.normal(size=(1, Sk, 1, d))
    v = np.eye(Sk).reshape(1, Sk, 1, Sk)
    scale = 0.8
    for causal in (False, True):
        p, lse = attn(q, k, v, causal=causal, scale=scale)
        p = p[0, :, 0, :]
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(p >= 0)
        for i in range(Sq):
            n = Sk if not causal else min(Sk, i + Sk - Sq + 1)
            assert np.all(p[i, n:] == 0.0)
            # ratio of two weights is e^{scale (q.k_a - q.k_b)}
            a, b = 0, n - 1
            sa = scale * float(q[0, i, 0] @ k[0, a, 0])
            sb = scale * float(q[0, i, 0] @ k[0, b, 0])
            assert abs(math.log(p[i, a] / p[i, b]) - (sa - sb)) < 1e-12
            # L_i = log sum_j e^{s_ij}: e^{s_ia - L_i} is the weight of key a
            assert abs(math.exp(sa - lse[0, 0, i]) - p[i, a]) < 1e-14


def check_permutation(attn):
    """Permuting keys and values together leaves O and L unchanged (non-causal)."""
    r = _rng(3)
    q = r.normal(size=(2, 4, 2, 6))
    k = r.normal(size=(2, 11, 2, 6))
    v = r.normal(size=(2, 11, 2, 3))
    perm = r.permutation(11)
    o1, l1 = attn(q, k, v, scale=0.5)
    o2, l2 = attn(q, k[:, perm], v[:, perm], scale=0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def check_key_shift(attn):
    """k_j -> k_j + w for every j: O unchanged, L_i -> L_i + scale q_i.w."""
    r = _rng(4)
    q = r.normal(size=(1, 5, 2, 4))
    k = r.normal(size=(1, 8, 2, 4))
    v = r.normal(size=(1, 8, 2, 2))
    w = r.normal(size=(4,))
    scale = 0.9
    for causal in (False, True):
        o1, l1 = attn(q, k, v, causal=causal, scale=scale)
        o2, l2 = attn(q, k + w, v, causal=causal, scale=scale)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        shift = scale * np.einsum("bihd,d->bhi", q, w)
        np.testing.assert_allclose(l2 - l1, shift, rtol=0, atol=1e-12)


def check_causal_row0(attn):
    """Sq = Sk causal: query 0 sees key 0 only: O_0 = V_0, L_0 = scale q_0.k_0."""
    r = _rng(5)
    q = r.normal(size=(1, 6, 3, 4))
    k = r.normal(size=(1, 6, 3, 4))
    v = r.normal(size=(1, 6, 3, 5))
    o, lse = attn(q, k, v, causal=True, scale=0.7)
    for h in range(3):
        np.testing.assert_allclose(o[0, 0, h], v[0, 0, h], rtol=0, atol=1e-14)
        assert abs(lse[0, h, 0] - 0.7 * float(q[0, 0, h] @ k[0, 0, h])) < 1e-13


def check_causal_as_truncation(attn):
    """Bottom-right causal row i equals a non-causal problem over keys 0..i+Sk-Sq;
    rows with no visible key give O = 0 and L = -inf."""
    r = _rng(6)
    for Sq, Sk in ((5, 5), (3, 8), (8, 3)):
        q = r.normal(size=(1, Sq, 2, 4))
        k = r.normal(size=(1, Sk, 1, 4))
        v = r.normal(size=(1, Sk, 1, 3))
        o, lse = attn(q, k, v, causal=True, scale=0.6)
        for i in range(Sq):
            n = min(Sk, i + Sk - Sq + 1)
            if n <= 0:
                assert np.all(o[0, i] == 0.0) and np.all(lse[0, :, i] == -np.inf)
                continue
            o1, l1 = attn(q[:, i:i + 1], k[:, :n], v[:, :n], causal=False, scale=0.6)
            np.testing.assert_allclose(o[0, i], o1[0, 0], rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[0, :, i], l1[0, :, 0], rtol=0, atol=1e-14)


def check_gqa_equals_mha(attn):
    """Query head h reads kv head h / ratio: same as MHA with K/V repeated."""
    r = _rng(7)
    Hq, Hkv = 6, 2
    q = r.normal(size=(2, 4, Hq, 5))
    k = r.normal(size=(2, 7, Hkv, 5))
    v = r.normal(size=(2, 7, Hkv, 3))
    for causal in (False, True):
        o1, l1 = attn(q, k, v, causal=causal, scale=0.4)
        o2, l2 = attn(q, np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2), causal=causal, scale=0.4)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-15)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-15)


def _brute(q, k, v, causal, scale):
    """Pure-Python loops over the definition (tiny inputs only)."""
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, dv = v.shape
    o = [[[[0.0] * dv for _ in range(Hq)] for _ in range(Sq)] for _ in range(B)]
    lse = [[[0.0] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for i in range(Sq):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                keys = [j for j in range(Sk) if (not causal) or j <= i + Sk - Sq]
                if not keys:
                    lse[b][h][i] = -math.inf
                    continue
                s = {j: scale * sum(float(q[b, i, h, c]) * float(k[b, j, g, c]) for c in range(d)) for j in keys}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in keys)
                for c in range(dv):
                    o[b][i][h][c] = sum(math.exp(s[j] - m) * float(v[b, j, g, c]) for j in keys) / z
                lse[b][h][i] = m + math.log(z)
    return np.array(o), np.array(lse)


def check_brute_force(attn):
    r = _rng(8)
    for causal in (False, True):
        q = r.normal(size=(2, 3, 4, 5))
        k = r.normal(size=(2, 6, 2, 5))
        v = r.normal(size=(2, 6, 2, 3))
        o, lse = attn(q, k, v, causal=causal, scale=0.45)
        ob, lb = _brute(q, k, v, causal, 0.45)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


def check_large_scores_stable(attn):
    """Scores in the hundreds (natural units) stay finite and exact: the
    stable softmax subtracts the row maximum."""
    q = np.array([[[[30.0]]]])
    k = np.array([10.0, 20.0, 30.0]).reshape(1, 3, 1, 1)
    v = np.array([1.0, 2.0, 3.0]).reshape(1, 3, 1, 1)
    o, lse = attn(q, k, v, scale=1.0)  # scores 300, 600, 900
    w = np.exp(np.array([-600.0, -300.0, 0.0]))
    assert abs(o[0, 0, 0, 0] - float(w @ np.array([1, 2, 3.0]) / w.sum())) < 1e-13
    assert abs(lse[0, 0, 0] - (900.0 + math.log(w.sum()))) < 1e-12


ALL_CHECKS = [check_worked_example, check_uniform_scores, check_probabilities, check_permutation,
              check_key_shift, check_causal_row0, check_causal_as_truncation, check_gqa_equals_mha,
              check_brute_force, check_large_scores_stable]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.attn_fwd)


# ----------------------------------------------------------------------------
# pins of the pages' online algebra (oracle.online)
# ----------------------------------------------------------------------------

def test_merge_figure_intermediates():
    """The block states and the merge of the worked example's figure."""
    g = json.load(open(os.path.join(GOLDEN, "online_merge_49_15.json")))
    x = np.log(np.array(g["exp_scores"], dtype=np.float64))
    vals = np.array(g["values"], dtype=np.float64)
    sa = online.block_state(x[:2], vals[:2])
    sb = online.block_state(x[2:], vals[2:])
    for st, gb in ((sa, g["block_a"]), (sb, g["block_b"])):
        assert abs(st[0] - math.log(gb["m_is_log_of"])) < 1e-15
        assert abs(st[1] - gb["l"]) < 1e-15
        assert abs(float(st[2][0]) - gb["u"]) < 1e-15
    m = max(sa[0], sb[0])
    assert abs(math.exp(sa[0] - m) - g["block_a"]["merge_factor"]) < 1e-15
    assert abs(math.exp(sb[0] - m) - g["block_b"]["merge_factor"]) < 1e-15
    merged = online.merge(sa, sb)
    assert abs(merged[0] - math.log(g["merged"]["m_is_log_of"])) < 1e-15
    assert abs(merged[1] - g["merged"]["l"]) < 1e-15
    assert abs(float(merged[2][0]) - g["merged"]["u"]) < 1e-15
    o, lse = online.finish(merged)
    assert abs(float(o[0]) - 49 / 15) < 1e-15
    assert abs(lse - math.log(15)) < 1e-14
    # averaging the two blocks' own outputs is not the answer (the page warns)
    naive = 0.5 * (sa[2][0] / sa[1] + sb[2][0] / sb[1])
    assert abs(naive - 49 / 15) > 0.1


@pytest.mark.parametrize("tau", [0.0, 8.0, math.inf])
def test_conditional_scan_worked_example(tau):
    """Two blocks of the worked example, scale 1: the kept-reference (tau=8)
    and always-rescale (tau=0) scans both give 49/15; tau=0 rescales once by
    the page's factor 1/4 = 2^delta with delta = (log 2 - log 8) * log2(e) = -2."""
    x = np.log(np.array([1.0, 2.0, 4.0, 8.0]))
    vals = np.array([1.0, 2.0, 3.0, 4.0])
    o, lse, n = online.conditional_scan(x, vals, block=2, scale=1.0, tau=tau)
    assert abs(float(o[0]) - 49 / 15) < 1e-14
    assert abs(lse - math.log(15)) < 1e-14
    assert n == (1 if tau == 0.0 else 0)


def _wide_range_row(r, n, d, dv, spread):
    q = r.normal(size=d) * 4.0
    k = r.normal(size=(n, d)) + np.linspace(0.0, spread, n)[:, None]
    v = r.normal(size=(n, dv))
    return q, k, v


@pytest.mark.parametrize("block", [1, 3, 16, 128])
@pytest.mark.parametrize("tau", [0.0, 8.0, math.inf])
def test_scans_reach_definition(block, tau):
    """flash_scan (Algorithm 1) and conditional_scan equal the definition on
    rows whose maximum keeps growing (keys offset 0 -> 12 along the sequence,
    q ~ 4 N(0,1)), with and without a causal prefix."""
    r = _rng(100 + block)
    d, dv, n = 24, 5, 300
    scale = 1 / math.sqrt(d)
    total_rescales = 0
    for trial in range(4):
        q, k, v = _wide_range_row(r, n, d, dv, 12.0)
        valid = np.ones(n, dtype=bool)
        if trial % 2:
            valid[n - 37:] = False  # a causal-style prefix
        nvis = int(valid.sum())
        o_ref, l_ref = oracle.attn_fwd(q.reshape(1, 1, 1, d), k[:nvis].reshape(1, nvis, 1, d),
                                       v[:nvis].reshape(1, nvis, 1, dv), scale=scale)
        raw = k @ q
        o1, l1 = online.flash_scan(raw * scale, v, block, valid)
        np.testing.assert_allclose(o1, o_ref[0, 0, 0], rtol=1e-12, atol=1e-12)
        assert abs(l1 - l_ref[0, 0, 0]) < 1e-10
        o2, l2, nres = online.conditional_scan(raw, v, block, scale, tau, valid)
        np.testing.assert_allclose(o2, o_ref[0, 0, 0], rtol=1e-12, atol=1e-12)
        assert abs(l2 - l_ref[0, 0, 0]) < 1e-10
        total_rescales += nres
    if tau == 8.0 and block >= 16:
        assert total_rescales > 0  # the wide range really crosses tau


def test_bf16_bits_decode_exactly():
    """The bf16 entry equals the float64 entry on the decoded values, bit for bit."""
    w = synthetic.Workload("t", 1, 4, 2, 33, 47, 16, 8, True, seed=11)
    q, k, v = w.generate()
    o1, l1 = oracle.attn_fwd(q, k, v, causal=True)
    f = synthetic.bf16_bits_to_f64
    o2, l2 = oracle.attn_fwd(f(q), f(k), f(v), causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_row_subset_matches_full():
    w = synthetic.Workload("t", 2, 4, 1, 40, 29, 16, 16, True, seed=12)
    q, k, v = w.generate()
    o, l = oracle.attn_fwd(q, k, v, causal=True)
    r = _rng(9)
    b, i, h = r.integers(0, 2, 50), r.integers(0, 40, 50), r.integers(0, 4, 50)
    rows = oracle.row_ids(b, i, h, 40, 4)
    o2, l2 = oracle.attn_fwd(q, k, v, causal=True, rows=rows)
    assert np.array_equal(o2, o[b, i, h]) and np.array_equal(l2, l[b, h, i])


def test_matches_torch_sdpa_float64():
    """torch float64 SDPA (+ logsumexp of the scaled scores) on CPU."""
    torch = pytest.importorskip("torch")
    r = _rng(10)
    for (B, Sq, Sk, Hq, Hkv, d, dv, causal) in [(2, 33, 33, 4, 4, 16, 16, False), (1, 17, 40, 6, 2, 8, 12, True),
                                                (2, 20, 20, 8, 1, 32, 16, True)]:
        q = r.normal(size=(B, Sq, Hq, d))
        k = r.normal(size=(B, Sk, Hkv, d))
        v = r.normal(size=(B, Sk, Hkv, dv))
        scale = 1 / math.sqrt(d)
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
        qt = torch.from_numpy(q).transpose(1, 2)
        kt = torch.from_numpy(np.repeat(k, Hq // Hkv, axis=2)).transpose(1, 2)
        vt = torch.from_numpy(np.repeat(v, Hq // Hkv, axis=2)).transpose(1, 2)
        mask = None
        if causal:
            i = torch.arange(Sq)[:, None]
            j = torch.arange(Sk)[None, :]
            mask = j <= i + Sk - Sq
        ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(o, ot.transpose(1, 2).numpy(), rtol=0, atol=1e-12)
        s = (qt @ kt.transpose(-1, -2)) * scale
        if mask is not None:
            s = s.masked_fill(~mask, -math.inf)
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# planted mistakes: each mutated copy of the oracle must fail some pin
# ----------------------------------------------------------------------------

MUTANTS = {
    "scale dropped": ("s[j] = J->scale * acc;", "s[j] = acc;"),
    "causal off by one": ("nvis = last + 1 < Sk ? last + 1 : Sk;", "nvis = last < Sk ? last : Sk;"),
    "top-left causal": ("int64_t last = i + Sk - Sq;", "int64_t last = i;"),
    "kv head modulo": ("const int64_t kvh = h / (J->Hq / J->Hkv);", "const int64_t kvh = h % J->Hkv;"),
    "lse without max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "no normalisation": ("o_row[c] /= l;", "o_row[c] /= 1.0;"),
    "max not subtracted": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "key/value index swapped": ("o_row[c] += s[j] * elem_at(J->v, voff + c, J->elem);",
                                "o_row[c] += s[nvis - 1 - j] * elem_at(J->v, voff + c, J->elem);"),
    "first key skipped": ("for (int64_t j = 1; j < nvis; ++j)\n    if (s[j] > m) m = s[j];",
                          "for (int64_t j = 1; j < nvis; ++j)\n    if (s[j] > m) m = s[j];\n  s[0] = -INFINITY;"),
    "empty row lse zero": ("*lse_out = -INFINITY;", "*lse_out = 0.0;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    path_c = os.path.join(mutant_dir, re.sub(r"\W+", "_", name) + ".c")
    path_so = path_c[:-2] + ".so"
    open(path_c, "w").write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", path_so, path_c, "-lm", "-lpthread"])
    lib = oracle.load_library(path_so)

    def attn(*a, **kw):
        return oracle.attn_fwd(*a, lib=lib, **kw)

    failed = []
    for check in ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(attn)
        except Exception:  # any failure of the check counts
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
