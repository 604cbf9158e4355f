"""Pins of the oracle's backward (``oracle.attn_bwd``) to facts other than
itself, and planted mistakes that each must fail one of them.

Pinned facts:
* central finite differences of the loss L = sum(dO * O), with O from the
  oracle's forward (a different code path: the forward never sees dO), on
  small problems with causal masks, Sq != Sk, GQA sharing and empty rows;
* torch float64 autograd through ``scaled_dot_product_attention`` with an
  explicit bottom-right mask and repeated K/V heads (a library routine);
* closed forms: with q = 0 every visible score is equal, so dK = 0 and dV_j is
  the sum over the rows i that see key j of dO_i / n_i (n_i the row's visible
  count); with all keys equal, the softmax-Jacobian rows sum to zero, so dQ = 0.
"""
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle


def loss(q, k, v, g, causal, scale):
    o, _ = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, threads=2)
    return float(np.sum(np.nan_to_num(o) * g))


CASES = [
    # B, Sq, Sk, Hq, Hkv, dqk, dv, causal
    (1, 5, 7, 2, 1, 4, 3, True),
    (1, 6, 6, 2, 2, 3, 3, False),
    (2, 7, 4, 4, 2, 3, 2, True),    # Sq > Sk: rows with no visible key
    (1, 4, 9, 3, 1, 5, 4, False),
]


def make(case, seed):
    B, Sq, Sk, Hq, Hkv, dqk, dv, causal = case
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Sq, Hq, dqk))
    k = rng.standard_normal((B, Sk, Hkv, dqk))
    v = rng.standard_normal((B, Sk, Hkv, dv))
    g = rng.standard_normal((B, Sq, Hq, dv))
    return q, k, v, g, causal


def pin_finite_differences(bwd):
    for n, case in enumerate(CASES):
        q, k, v, g, causal = make(case, 100 + n)
        scale = 0.7
        dq, dk, dv = bwd(q, k, v, g, causal, scale)
        rng = np.random.default_rng(n)
        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(6):
                idx = tuple(int(rng.integers(0, s)) for s in x.shape)
                h = 1e-5
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = dict(q=q, k=k, v=v)
                args_m = dict(q=q, k=k, v=v)
                args_p[name], args_m[name] = xp, xm
                fd = (loss(args_p["q"], args_p["k"], args_p["v"], g, causal, scale)
                      - loss(args_m["q"], args_m["k"], args_m["v"], g, causal, scale)) / (2 * h)
                assert abs(fd - grad[idx]) <= 1e-6 * (1 + abs(fd)), (case, name, idx, fd, grad[idx])


def pin_torch_autograd(bwd):
    torch = pytest.importorskip("torch")
    for n, case in enumerate(CASES):
        q, k, v, g, causal = make(case, 200 + n)
        B, Sq, Sk, Hq, Hkv, dqk, dv, _ = case
        scale = 0.5
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        ratio = Hq // Hkv
        qh = tq.permute(0, 2, 1, 3)
        kh = tk.permute(0, 2, 1, 3).repeat_interleave(ratio, dim=1)
        vh = tv.permute(0, 2, 1, 3).repeat_interleave(ratio, dim=1)
        s = scale * qh @ kh.transpose(-1, -2)
        if causal:
            i = torch.arange(Sq)[:, None]
            j = torch.arange(Sk)[None, :]
            s = s.masked_fill(~(j <= i + Sk - Sq), float("-inf"))
        p = torch.softmax(s, dim=-1).nan_to_num(0.0)  # rows with no visible key: 0
        o = (p @ vh).permute(0, 2, 1, 3)
        (o * torch.tensor(g)).sum().backward()
        dq, dk, dv_ = bwd(q, k, v, g, causal, scale)
        for want, got in ((tq.grad, dq), (tk.grad, dk), (tv.grad, dv_)):
            assert np.allclose(want.numpy(), got, atol=1e-11, rtol=1e-10), case


def pin_closed_forms(bwd):
    rng = np.random.default_rng(7)
    B, Sq, Sk, Hq, Hkv, d = 1, 6, 5, 2, 1, 3
    for causal in (False, True):
        q = np.zeros((B, Sq, Hq, d))
        k = rng.standard_normal((B, Sk, Hkv, d))
        v = rng.standard_normal((B, Sk, Hkv, d))
        g = rng.standard_normal((B, Sq, Hq, d))
        dq, dk, dv = bwd(q, k, v, g, causal, 1.0)
        assert np.allclose(dk, 0.0, atol=1e-14)
        want = np.zeros_like(dv)
        for h in range(Hq):
            for i in range(Sq):
                nvis = Sk if not causal else max(0, min(Sk, i + Sk - Sq + 1))
                for j in range(nvis):
                    want[0, j, 0] += g[0, i, h] / nvis
        assert np.allclose(dv, want, atol=1e-14)
        # all keys equal: dQ = scale * sum_j dS_ij k = 0
        k_eq = np.repeat(k[:, :1], Sk, axis=1)
        q2 = rng.standard_normal((B, Sq, Hq, d))
        dq2, _, _ = bwd(q2, k_eq, v, g, causal, 1.0)
        assert np.allclose(dq2, 0.0, atol=1e-13)


PINS = [pin_finite_differences, pin_torch_autograd, pin_closed_forms]


def oracle_bwd(lib=None):
    return lambda q, k, v, g, causal, scale: oracle.attn_bwd(q, k, v, g, causal=causal, scale=scale, threads=2,
                                                             lib=lib)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_backward_pins(pin):
    pin(oracle_bwd())


def test_bf16_inputs_decode_like_doubles():
    rng = np.random.default_rng(3)
    import synthetic
    bits = [synthetic.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
            for s in ((1, 9, 2, 8), (1, 11, 1, 8), (1, 11, 1, 8), (1, 9, 2, 8))]
    dbl = [synthetic.bf16_bits_to_f64(b) for b in bits]
    a = oracle.attn_bwd(*bits, causal=True, threads=2)
    b = oracle.attn_bwd(*dbl, causal=True, threads=2)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ----------------------------------------------------------------------------
# planted mistakes: each mutated copy of the backward must fail some pin
# ----------------------------------------------------------------------------

MUTANTS = {
    "D term dropped": ("const double ds = p[j] * (dp[j] - D);", "const double ds = p[j] * dp[j];"),
    "dK without scale": ("J->dk[koff + c] += J->scale * ds * elem_at(J->q, qoff + c, J->elem);",
                         "J->dk[koff + c] += ds * elem_at(J->q, qoff + c, J->elem);"),
    "dV from dP": ("J->dvv[voff + c] += p[j] * elem_at(J->dout, ooff + c, J->elem);",
                   "J->dvv[voff + c] += dp[j] * elem_at(J->dout, ooff + c, J->elem);"),
    "dQ from Q": ("dq_row[c] += J->scale * ds * elem_at(J->k, koff + c, J->elem);",
                  "dq_row[c] += J->scale * ds * elem_at(J->q, qoff + c, J->elem);"),
    "D as sum of P": ("D += p[j] * acc;", "D += p[j];"),
    "wrong shared head": ("for (int64_t h = kvh * ratio; h < (kvh + 1) * ratio; ++h) {",
                          "for (int64_t h = kvh; h < J->Hq; h += J->Hkv) {"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_bwd_mutants_")
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
    failed = []
    for pin in PINS:
        try:
            pin(oracle_bwd(lib))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
