"""The polynomial exp2 of the optional FMA-pipe path: coefficients and accuracy.

The pages report that a degree-3 polynomial with Cody-Waite reduction matches
the hardware exponential to within one bf16 unit on 99 % of inputs
("FlashAttention-4 wiki", "Core methods").  Checked here in a float32
simulation of the kernel's steps against exact 2^x, both rounded to bf16."""
import os
import re

import numpy as np

from exact_attention_forward_08_gb300 import exp2_poly

KERNEL = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "exact_attention_forward_08_gb300",
                      "csrc", "fa_kernel.cuh")


def kernel_coefficients():
    src = open(KERNEL).read()
    return [float(re.search(rf"kExp2C{i} = ([0-9.e+-]+)f;", src).group(1)) for i in range(4)]


def test_kernel_constants_are_the_fit():
    fitted = exp2_poly.coefficients_f32()
    for k, f in zip(kernel_coefficients(), fitted):
        assert np.float32(k) == np.float32(f)
    assert exp2_poly.max_rel_error(np.array(fitted)) < 1e-4


def to_bf16(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.int64)


def simulate(x):
    """The kernel's steps in float32 (each fused multiply-add rounded once)."""
    f32 = np.float32
    c = [f32(v) for v in kernel_coefficients()]
    xc = np.maximum(x.astype(f32), f32(-126.0))
    magic = f32(12582912.0)
    t = (xc + magic).astype(f32)
    jf = (t - magic).astype(f32)
    f = (xc.astype(np.float64) - jf.astype(np.float64)).astype(f32)
    q = (c[3].astype(np.float64) * f + c[2]).astype(f32)
    q = (q.astype(np.float64) * f + c[1]).astype(f32)
    q = (q.astype(np.float64) * f + c[0]).astype(f32)
    bits = q.view(np.uint32).astype(np.uint64) + ((t.view(np.uint32).astype(np.uint64) << 23) & 0xFFFFFFFF)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_within_one_bf16_unit_on_99_percent():
    x = np.random.default_rng(0).uniform(-60.0, 8.0, 200000).astype(np.float32)
    y = simulate(x)
    exact = np.exp2(x.astype(np.float64)).astype(np.float32)
    d = np.abs(to_bf16(y) - to_bf16(exact))
    assert d.max() <= 1
    assert np.mean(d == 0) >= 0.95
    assert np.mean(d <= 1) >= 0.99
    # integers are exact; very negative inputs stay tiny and positive
    ints = np.arange(-120, 9, dtype=np.float32)
    assert np.array_equal(to_bf16(simulate(ints)), to_bf16(np.exp2(ints)))
    tiny = simulate(np.array([-126.0, -200.0, -1e30], np.float32))
    assert np.all(tiny >= 0) and np.all(tiny < 1e-37)
