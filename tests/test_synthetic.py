"""The seeded input generator: determinism, distribution and the recipes."""
import numpy as np

import synthetic


def test_deterministic_and_thread_independent(monkeypatch):
    a = synthetic.normal_bf16((3, 70000), seed=5, stream=1)
    b = synthetic.normal_bf16((3, 70000), seed=5, stream=1)
    assert np.array_equal(a, b)
    monkeypatch.setattr(synthetic, "_threads", lambda: 1)
    c = synthetic.normal_bf16((3, 70000), seed=5, stream=1)
    assert np.array_equal(a, c)
    d = synthetic.normal_bf16((3, 70000), seed=5, stream=2)
    assert not np.array_equal(a, d)


def test_standard_normal_moments():
    x = synthetic.bf16_bits_to_f64(synthetic.normal_bf16((1 << 20,), seed=1, stream=3))
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert abs(np.mean(np.abs(x) < 1.0) - 0.6827) < 3e-3


def test_bf16_rounding_round_trip():
    x = np.array([1.0, -2.5, 3.140625, 1e-3, 65504.0], dtype=np.float32)
    bits = synthetic.f32_to_bf16_bits(x)
    back = synthetic.bf16_bits_to_f32(bits)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8)
    # ties go to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert synthetic.f32_to_bf16_bits(np.array([1.0 + 2.0 ** -8], np.float32))[0] == 0x3F80


def test_offset_recipe_rises_along_sequence():
    k = synthetic.bf16_bits_to_f64(synthetic.normal_offset_bf16((2, 64, 4, 32), seed=4, stream=2, mul=1.0,
                                                                off_max=12.0))
    per_pos = k.mean(axis=(0, 2, 3))
    assert abs(per_pos[0]) < 0.5 and abs(per_pos[-1] - 12.0) < 0.5
    assert np.all(np.diff(np.convolve(per_pos, np.ones(8) / 8, mode="valid")) > -0.3)


def test_workload_table():
    w = synthetic.workloads()
    assert w["mha8k"].flops() == 4 * 4 * 16 * 8192 * 8192 * 128
    assert w["causal8k"].flops() == 2 * 4 * 16 * 8192 * 8192 * 128
    assert w["asym"].flops() == 2 * 2 * 16 * 16384 * 16384 * (192 + 128) / 2
    assert all(x.batch * x.seqlen_q == 32768 for n, x in w.items() if n.startswith("causal"))
