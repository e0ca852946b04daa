"""Pins of the oracle's low-rank key reconstruction: closed forms (rank one with a
unit coefficient, integer factors), the fp64 product within the bf16 and fp32
rounding bounds, the float32 -> bf16 rounding on hand values, and agreement
with the generator's independently written low-rank keys.  CPU only."""
import numpy as np

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS


def _bits(x):
    return orc.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_bf16_rounding_hand_values():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties to even gives 1.0 (0x3F80)
    assert _bits([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0]).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0]
    # 1 + 3*2^-8 lies between 1 + 2^-7 (0x3F81) and 1 + 2^-6 (0x3F82): tie, even mantissa wins (0x3F82)


def test_rank_one_unit_coefficient_returns_the_basis_row():
    rng = np.random.default_rng(0)
    e = _bits(rng.standard_normal((1, 16)))
    a = _bits(np.ones((5, 1)))
    out = orc.lowrank_keys(a, e)
    assert (out == e[0]).all()


def test_integer_factors_are_exact():
    rng = np.random.default_rng(1)
    a = rng.integers(-3, 4, size=(7, 4)).astype(np.float32)
    e = rng.integers(-3, 4, size=(4, 6)).astype(np.float32)
    out = orc.bf16_bits_to_f64(orc.lowrank_keys(_bits(a), _bits(e)))
    assert np.array_equal(out, a.astype(np.float64) @ e.astype(np.float64))


def test_close_to_the_exact_product():
    rng = np.random.default_rng(2)
    R = 32
    a_b = _bits(rng.standard_normal((64, R)))
    e_b = _bits(rng.standard_normal((R, 128)) / np.sqrt(R))
    a, e = orc.bf16_bits_to_f64(a_b), orc.bf16_bits_to_f64(e_b)
    exact = a @ e
    got = orc.bf16_bits_to_f64(orc.lowrank_keys(a_b, e_b))
    bound = 2.0 ** -8 * np.abs(exact) + R * 2.0 ** -24 * (np.abs(a) @ np.abs(e)) * 2 + 1e-30
    assert (np.abs(got - exact) <= bound).all()


def test_agrees_with_the_generated_low_rank_keys():
    w = WORKLOADS["lowrank_predict"].scaled(batch=1, ctx=(600, 600), window=24)
    K, _ = synth.gen_request_kv(w, 9, 0, 0, 600, None)
    coef, basis = synth.gen_lowrank_factors(w, 9, 0, 0, 600)
    for g in range(w.n_kv_heads):
        assert np.array_equal(orc.lowrank_keys(synth.bits(coef[g]), synth.bits(basis[g])), synth.bits(K[g]))
