"""Pins for the oracle's query / KV RMSNorm and partial RoPE (report §2.3.3:
each head's query and the KV entries are RMS-normalized before the core
attention; RoPE turns the last 64 dims of every query and KV entry vector,
and the core attention's output, to carry relative positions).  Each check
ties the oracle to something other than its own formula: closed forms,
rotation written as complex multiplication, invariances.  CPU only."""
import numpy as np
import pytest

from oracle import csa

RNG = np.random.default_rng(99)
D = 576


def test_rms_norm_closed_forms():
    g = RNG.random(D) + 0.5
    for c in (3.0, -0.25):
        x = np.full(D, c)
        assert np.allclose(csa.rms_norm(x, g, 0.0), np.sign(c) * g, rtol=0, atol=1e-15)
        assert np.allclose(csa.rms_norm(x, g, 1e-2), c / np.sqrt(c * c + 1e-2) * g, rtol=1e-15, atol=0)
    x = RNG.standard_normal((4, D)) * 7
    y = csa.rms_norm(x, np.ones(D), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    # scale invariance: a positive factor on x changes nothing (eps = 0)
    assert np.allclose(csa.rms_norm(5 * x, g, 0.0), csa.rms_norm(x, g, 0.0), rtol=1e-14, atol=1e-14)


def test_rope_is_complex_rotation_of_the_last_64_dims():
    x = RNG.standard_normal((3, D))
    pos = np.array([0, 17, 123456])
    y = csa.rope(x, pos, 10000.0)
    assert np.array_equal(y[:, :512], x[:, :512])
    z = x[:, 512::2] + 1j * x[:, 513::2]
    freq = 10000.0 ** (-np.arange(32) / 32.0)  # base^(-2i/64)
    zr = z * np.exp(1j * pos[:, None] * freq[None])
    assert np.allclose(y[:, 512::2], zr.real, atol=1e-12) and np.allclose(y[:, 513::2], zr.imag, atol=1e-12)
    assert np.array_equal(csa.rope(x, np.zeros(3), 10000.0), x)


def test_rope_group_properties():
    x = RNG.standard_normal((5, D))
    a, b = np.array([3, 40, 700, 9000, 65535]), np.array([11, -40, 5, 123, 1])
    assert np.allclose(csa.rope(csa.rope(x, a, 1e4), b, 1e4), csa.rope(x, a + b, 1e4), atol=1e-10)
    assert np.allclose(csa.rope(csa.rope(x, a, 1e4), -a, 1e4), x, atol=1e-10)
    # norm of every rotated pair is kept
    y = csa.rope(x, a, 1e4)
    assert np.allclose(np.hypot(y[:, 512::2], y[:, 513::2]), np.hypot(x[:, 512::2], x[:, 513::2]), rtol=1e-13)


def test_rope_dot_product_depends_on_offset_only():
    q, k = RNG.standard_normal(D), RNG.standard_normal(D)
    for t, s in [(100, 37), (5000, 4937), (1048576 + 90, 1048576 + 27)]:
        d = csa.rope(q[None], [t], 1e4)[0] @ csa.rope(k[None], [s], 1e4)[0]
        d0 = csa.rope(q[None], [63], 1e4)[0] @ k
        assert abs(d - d0) < 1e-9 * (np.abs(q) @ np.abs(k))


def _case(t, m=4, n_ent=6, W=5, shift=0):
    """One query at t over n_ent compressed entries and W window tokens, all
    positions moved by `shift`."""
    H = 3
    g = np.random.default_rng(7)
    q = g.standard_normal((H, D))
    comp = g.standard_normal((n_ent, D)) * 3
    win = g.standard_normal((W, D)) * 2
    qg, kg = g.random(D) + 0.5, g.random(D) + 0.5
    ent = csa.rope(csa.rms_norm(comp, kg, 1e-6), csa.entry_position(np.arange(n_ent), m) + shift, 1e4)
    wpos = np.arange(t - W + 1, t + 1) + shift
    return csa.attend_one_rope(q, t + shift, ent, None, win, wpos, 1 / 24, qg, kg, 1e-6, 1e4)


def test_rotated_attention_is_translation_invariant():
    """Moving the query and every key by the same offset changes nothing:
    RoPE makes the logits depend on offsets only, and the output's rotation
    back by t makes its RoPE dims relative too."""
    o0, l0 = _case(40)
    for shift in (1, 1000, 1048576):
        o1, l1 = _case(40, shift=shift)
        assert np.allclose(o1, o0, atol=1e-9) and np.allclose(l1, l0, atol=1e-9)


def test_rotated_attention_single_token():
    """Only the current token visible: the output is that token normalized
    with the KV gain (rotated by t, then back by t), for every head."""
    g = np.random.default_rng(8)
    k = g.standard_normal((1, D))
    kg = g.random(D) + 0.5
    q = g.standard_normal((2, D))
    o, _ = csa.attend_one_rope(q, 77, np.zeros((0, D)), None, k, [77], 0.1, np.ones(D), kg, 1e-6, 1e4)
    assert np.allclose(o, np.repeat(csa.rms_norm(k, kg, 1e-6), 2, 0), atol=1e-12)


def test_rotated_attention_equals_plain_attention_on_prepared_vectors():
    """attend_one_rope is the plain attention of the normalized, rotated
    query over the prepared keys, with the output turned back by -t: checked
    through the logits written out as per-pair complex products."""
    t, H, W = 30, 2, 4
    g = np.random.default_rng(9)
    q = g.standard_normal((H, D))
    win = g.standard_normal((W, D))
    wpos = np.arange(t - W + 1, t + 1)
    o, lse = csa.attend_one_rope(q, t, np.zeros((0, D)), None, win, wpos, 0.2, np.ones(D), np.ones(D), 0.0, 1e4)
    qn, wn = csa.rms_norm(q, np.ones(D), 0.0), csa.rms_norm(win, np.ones(D), 0.0)
    freq = 1e4 ** (-np.arange(32) / 32.0)
    zq = qn[:, 512::2] + 1j * qn[:, 513::2]
    zk = wn[:, 512::2] + 1j * wn[:, 513::2]
    # Re(conj(z_q e^{i t f}) z_k e^{i s f}) = Re(conj(z_q) z_k e^{i (s - t) f})
    rot = np.real(np.conj(zq)[:, None, :] * zk[None, :, :] * np.exp(1j * (wpos - t)[None, :, None] * freq)).sum(-1)
    logits = 0.2 * (qn[:, :512] @ wn[:, :512].T + rot)
    assert np.allclose(lse, np.log(np.exp(logits).sum(1)), atol=1e-12)
    p = np.exp(logits - lse[:, None])
    want_c = p @ wn[:, :512]
    zo = (p[:, :, None] * zk[None] * np.exp(1j * (wpos - t)[None, :, None] * freq)).sum(1)
    assert np.allclose(o[:, :512], want_c, atol=1e-12)
    assert np.allclose(o[:, 512::2], zo.real, atol=1e-12) and np.allclose(o[:, 513::2], zo.imag, atol=1e-12)
