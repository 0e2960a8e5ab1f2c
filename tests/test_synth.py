"""The seeded input generator: counter-based, order-free, bf16 round-to-nearest-even."""
import numpy as np

import synth


def test_counter_based_slices():
    full = synth.normal_f64(0, 7, 1000)
    part = synth.normal_f64(0, 7, 300, offset=500)
    np.testing.assert_array_equal(full[500:800], part)
    assert not np.array_equal(synth.normal_f64(0, 8, 1000), full)
    assert not np.array_equal(synth.normal_f64(1, 7, 1000), full)


def test_normal_moments():
    x = synth.normal_f64(3, 1, 400000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(np.mean(x ** 3)) < 0.02 and abs(np.mean(x ** 4) - 3.0) < 0.05


def test_bf16_rounding():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, 1.0 + 2 ** -9])
    u = synth.round_bf16(vals)
    # 1+2^-8 is a tie between 1 and 1+2^-7: goes to the even mantissa (1.0); 1+3*2^-8 goes up to 1+2^-6
    assert u.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x3F80]
    np.testing.assert_array_equal(synth.bf16_to_f64(u), [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0, 1.0])


def test_workload_recipe():
    Wg, W1, W2 = synth.ffn_weights(0, 64, 256)
    assert Wg.shape == (256, 64) and W2.shape == (64, 256) and Wg.dtype == np.uint16
    w = synth.bf16_to_f64(Wg)
    assert abs(w.std() - 0.02) < 0.001
    sc = synth.dim_scales(0, 64)
    assert sc.shape == (64,) and np.all(sc > 0)
    X = synth.prompt(0, 10, sc)
    x0 = synth.decode_input(0, 0, 2, sc)
    x1 = synth.decode_input(0, 1, 2, sc)
    assert X.shape == (10, 64) and x0.shape == (2, 64) and not np.array_equal(x0, x1)
    # same scale per column: the column spread follows c_d
    big = synth.bf16_to_f64(synth.prompt(0, 4000, sc))
    ratio = big.std(axis=0) / sc
    assert np.all(np.abs(ratio - 1.0) < 0.1)
