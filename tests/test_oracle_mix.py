"""Pins of the oracle's MIMO head mixer (the fused epilogue's reference): out
head g = sum_h W[g, h] Re(y) head h, checked against a loop written out
element by element on a tiny case, and against what its special cases must
give: the identity (the pages' initialisation) returns Re(y) itself, a
permutation permutes the heads, a multiple of the identity scales, and the
map is linear in W and in y."""
import numpy as np

from oracle import head_mix


def _y(shape, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) + 1j * rng.standard_normal(shape)


def test_loop_on_a_tiny_case():
    y = _y((2, 3, 4, 5), 1)
    W = np.random.default_rng(2).standard_normal((4, 4))
    out = head_mix(y, W)
    for b in range(2):
        for t in range(3):
            for g in range(4):
                for d in range(5):
                    want = sum(W[g, h] * y[b, t, h, d].real for h in range(4))
                    assert abs(out[b, t, g, d] - want) < 1e-12


def test_identity_permutation_scaling():
    y = _y((1, 7, 16, 8), 3)
    assert np.array_equal(head_mix(y, np.eye(16)), y.real)
    perm = np.random.default_rng(4).permutation(16)
    P = np.eye(16)[perm]  # row g picks head perm[g]
    assert np.array_equal(head_mix(y, P), y.real[:, :, perm, :])
    assert np.allclose(head_mix(y, 2.5 * np.eye(16)), 2.5 * y.real, rtol=0, atol=1e-13)


def test_linear_in_w_and_y():
    y1, y2 = _y((2, 5, 6, 4), 5), _y((2, 5, 6, 4), 6)
    rng = np.random.default_rng(7)
    W1, W2 = rng.standard_normal((6, 6)), rng.standard_normal((6, 6))
    assert np.allclose(head_mix(y1, W1 + W2), head_mix(y1, W1) + head_mix(y1, W2), atol=1e-12)
    assert np.allclose(head_mix(y1 + y2, W1), head_mix(y1, W1) + head_mix(y2, W1), atol=1e-12)
    # only the real part of y enters
    assert np.array_equal(head_mix(y1, W1), head_mix(y1.real + 0j, W1))
