"""The seeded input generator (CPU): determinism, rounding, masks and the peaked recipe."""
import numpy as np

from memory_efficient_exact_gb300 import inputs as I


def test_round_bf16_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9, -2.5, 0.0], dtype=np.float32)
    r = I.round_bf16(x)
    # 1 + 2^-8 lies half-way between 1 and 1 + 2^-7: ties go to the even mantissa (1)
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == np.float32(1.0 + 2.0 ** -7) and r[3] == -2.5 and r[4] == 0.0
    # every rounded value has a zero low half-word
    assert np.all((I.round_bf16(np.random.default_rng(0).standard_normal(1000).astype(np.float32))
                   .view(np.uint32) & 0xFFFF) == 0)


def test_workload_draws_are_deterministic_and_prefix_stable():
    a = I.make_hw(64, 16, 50, 5, "bf16")
    b = I.make_hw(64, 16, 50, 5, "bf16")
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    # a shorter draw is the prefix of a longer one (row blocks of the same streams)
    c = I.make_hw(32, 16, 50, 5, "bf16")
    assert np.array_equal(c[0], a[0][:32]) and np.array_equal(c[1], a[1])


def test_masks():
    y = I.make_labels(100, 7, 3, "frac", 0.1)
    assert np.sum(y == I.IGNORE_INDEX) == 10 and np.all((y == I.IGNORE_INDEX) | ((y >= 0) & (y < 7)))
    y = I.make_labels(100, 7, 3, "seqhead", n=4, seq_len=25)
    assert np.all(y.reshape(4, 25)[:, :4] == I.IGNORE_INDEX) and np.all(y.reshape(4, 25)[:, 4:] >= 0)


def test_peaked_recipe():
    T, d, V = 64, 128, 300
    H, W, y = I.make_peaked(T, d, V, 9, "bf16", 8.0, 30.0, 40.0, frac=0.25,
                            copies=((7, 3),), labels=np.full(T, 3))
    assert np.array_equal(W[7], W[3])
    assert np.sum(y == I.IGNORE_INDEX) == T // 4 and np.all(y[y != I.IGNORE_INDEX] == 3)
    assert np.all((H.view(np.uint32) & 0xFFFF) == 0) and np.all((W.view(np.uint32) & 0xFFFF) == 0)
    # the lift raises the tokens' dot products with their label row by a_t ~ U[30, 40] on
    # average, over a background of standard deviation about sigma_z = 8 (widened a little,
    # about a_t / sqrt(d), by the nudge itself)
    Z = H.astype(np.float64) @ W.astype(np.float64).T
    assert abs(Z[:, 3].mean() - 35.0) < 4.0 and 7.5 < np.std(np.delete(Z, [3, 7], axis=1)) < 9.5
    H2, W2, y2 = I.make_peaked(T, d, V, 9, "bf16", 8.0, 30.0, 40.0, frac=0.25,
                               copies=((7, 3),), labels=np.full(T, 3))
    assert np.array_equal(H, H2) and np.array_equal(W, W2) and np.array_equal(y, y2)
