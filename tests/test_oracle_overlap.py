"""Pins for the oracle's overlapping compression (report §2.3.1: two KV sets
C_a, C_b with weights Z_a, Z_b; §2.3.2: HCA has no overlap): special cases
that reduce to the plain compressor or to closed forms.  CPU only."""
import numpy as np

from oracle import csa

RNG = np.random.default_rng(77)
D = 24


def _streams(n, m, scale_b=1.0):
    return (RNG.standard_normal((n, D)), RNG.standard_normal((n, D)) * 2, RNG.standard_normal((m, D)) * 0.1,
            RNG.standard_normal((n, D)), RNG.standard_normal((n, D)) * 2 * scale_b, RNG.standard_normal((m, D)) * 0.1)


def test_without_the_previous_block_it_is_the_plain_compressor():
    # C_b's gates at -inf give C_b no weight: the plain compressor of C_a
    m, n = 4, 40
    ka, ga, ba, kb, gb, bb = _streams(n, m)
    gb[:] = -np.inf
    assert np.allclose(csa.compress_overlap(ka, ga, ba, kb, gb, bb, m), csa.compress(ka, ga, ba, m), atol=1e-14)
    # entry 0 never has a previous block
    ka, ga, ba, kb, gb, bb = _streams(n, m)
    assert np.allclose(csa.compress_overlap(ka, ga, ba, kb, gb, bb, m)[0], csa.compress(ka, ga, ba, m)[0],
                       atol=1e-14)


def test_previous_block_alone_when_it_dominates():
    # C_a's gates at -inf (from entry 1 on): entry j is the plain compressor of
    # C_b over block j - 1
    m, n = 4, 40
    ka, ga, ba, kb, gb, bb = _streams(n, m)
    ga[m:] = -np.inf
    out = csa.compress_overlap(ka, ga, ba, kb, gb, bb, m)
    want = csa.compress(kb, gb, bb, m)
    assert np.allclose(out[1:], want[:-1], atol=1e-14)


def test_identical_tokens_and_weights_sum_to_one():
    m, n = 4, 32
    tok = RNG.standard_normal(D)
    ka, ga, ba, kb, gb, bb = _streams(n, m)
    out = csa.compress_overlap(np.tile(tok, (n, 1)), ga, ba, np.tile(tok, (n, 1)), gb, bb, m)
    assert np.allclose(out, np.tile(tok, (n // m, 1)), atol=1e-13)
    # all-ones values: the output is the sum of the weights
    ones = np.ones((n, D))
    assert np.allclose(csa.compress_overlap(ones, ga, ba, ones, gb, bb, m), 1.0, atol=1e-14)


def test_m1_closed_form():
    # m = 1: entry j mixes C_a[j] and C_b[j - 1] with a two-way softmax
    n = 12
    ka, ga, ba, kb, gb, bb = _streams(n, 1)
    out = csa.compress_overlap(ka, ga, ba, kb, gb, bb, 1)
    assert np.allclose(out[0], ka[0])
    for j in range(1, n):
        za, zb = ga[j] + ba[0], gb[j - 1] + bb[0]
        wa = 1.0 / (1.0 + np.exp(zb - za))
        assert np.allclose(out[j], wa * ka[j] + (1 - wa) * kb[j - 1], atol=1e-13)


def test_equal_logits_average_both_blocks():
    m, n = 4, 16
    ka, _, _, kb, _, _ = _streams(n, m)
    z = np.zeros((n, D))
    out = csa.compress_overlap(ka, z, np.zeros((m, D)), kb, z, np.zeros((m, D)), m)
    for j in range(1, n // m):
        want = (ka[j * m:(j + 1) * m].sum(0) + kb[(j - 1) * m:j * m].sum(0)) / (2 * m)
        assert np.allclose(out[j], want, atol=1e-14)
