"""Pins for the oracle's compressor (not the GPU): the pages' worked example and
properties the equations fix."""
import numpy as np
import pytest

from oracle import csa2_oracle as O


def _rng(seed):
    return np.random.default_rng(seed)


def test_worked_example_overlap(golden):
    g = golden("compressor_worked_example.json")
    m, c = g["m"], g["c"]
    Ca = np.array(g["Ca_rows"], dtype=float)
    Cb = np.array(g["Cb_rows"], dtype=float)
    Z = np.zeros_like(Ca)
    y = O.compress(Ca, Z, m, np.zeros((m, c)), Cb, Z, np.zeros((m, c)))
    np.testing.assert_allclose(y, np.array(g["expected"]), rtol=0, atol=1e-15)


def test_m1_is_identity():
    # m = 1: a softmax over one position is 1, so each entry is its token.
    r = _rng(1)
    Ca = r.normal(size=(37, 16))
    Za = r.normal(size=(37, 16)) * 5
    np.testing.assert_array_equal(O.compress(Ca, Za, 1), Ca)


def test_equal_logits_give_mean():
    r = _rng(2)
    m = 4
    Ca = r.normal(size=(4 * m, 8))
    Za = np.full_like(Ca, 3.25)
    y = O.compress(Ca, Za, m)
    np.testing.assert_allclose(y, Ca.reshape(4, m, 8).mean(axis=1), rtol=1e-14, atol=1e-14)


def test_dominant_logit_selects_row():
    r = _rng(3)
    m = 4
    Ca = r.normal(size=(2 * m, 5))
    Za = np.zeros_like(Ca)
    Za[1] = 60.0   # block 0, position 1 wins in every channel
    Za[6] = 60.0   # block 1, position 2
    y = O.compress(Ca, Za, m)
    np.testing.assert_allclose(y[0], Ca[1], rtol=0, atol=8 * np.exp(-60))
    np.testing.assert_allclose(y[1], Ca[6], rtol=0, atol=8 * np.exp(-60))


def test_bias_shifts_weights_per_channel():
    # A bias of +50 on in-block position j for channel ch makes that channel copy
    # position j's value; other channels are untouched.
    r = _rng(4)
    m, c = 2, 4
    Ca = r.normal(size=(3 * m, c))
    Za = np.zeros_like(Ca)
    Ba = np.zeros((m, c))
    Ba[1, 2] = 50.0
    y = O.compress(Ca, Za, m, Ba)
    for i in range(3):
        assert abs(y[i, 2] - Ca[m * i + 1, 2]) < 1e-20 + 4 * np.exp(-50)
        np.testing.assert_allclose(y[i, [0, 1, 3]], Ca[m * i:m * i + m][:, [0, 1, 3]].mean(0), rtol=1e-14)


def test_first_block_has_no_history_mass():
    r = _rng(5)
    m, c, n = 4, 6, 16
    Ca, Cb, Za, Zb = (r.normal(size=(n, c)) for _ in range(4))
    Ba, Bb = r.normal(size=(m, c)), r.normal(size=(m, c))
    y = O.compress(Ca, Za, m, Ba, Cb, Zb, Bb)
    # block 0 must equal the history-free softmax of block 0 alone
    y0 = O.compress(Ca[:m], Za[:m], m, Ba)
    np.testing.assert_allclose(y[0], y0[0], rtol=1e-14, atol=1e-15)
    # and must not change when the (absent) history is made huge
    y_big = O.compress(Ca, Za, m, Ba, Cb * 1e6, Zb + 100, Bb)
    np.testing.assert_array_equal(y[0], y_big[0])


def test_second_block_reads_previous_cb():
    # entry 1 mixes block 1's C^a with block 0's C^b (not block 1's C^b)
    m, c = 2, 1
    Ca = np.array([[0.], [0.], [1.], [1.]])
    Cb = np.array([[5.], [5.], [9.], [9.]])
    Z = np.zeros_like(Ca)
    y = O.compress(Ca, Z, m, None, Cb, Z, None)
    assert y[1, 0] == pytest.approx(3.0, abs=1e-15)   # mean of 1, 1, 5, 5


def test_two_overlap_formulations_agree():
    # DSA-to-CSA/HCA eqs. 11-12 vs the Attention-evolution page's overlap_transform:
    # C^a = upper half, C^b = lower half of the 2d projection, same for logits/APE.
    r = _rng(6)
    m, d, G = 4, 8, 7
    kv = r.normal(size=(G * m, 2 * d))
    gate = r.normal(size=(G * m, 2 * d))
    ape = r.normal(size=(m, 2 * d)) * 0.1
    y1 = O.compress_overlap_transform(kv, gate, ape, m)
    y2 = O.compress(kv[:, d:], gate[:, d:], m, ape[:, d:], kv[:, :d], gate[:, :d], ape[:, :d])
    np.testing.assert_allclose(y1, y2, rtol=1e-13, atol=1e-14)


def test_chunked_equals_whole_with_carried_state():
    r = _rng(7)
    m, c = 4, 5
    n_ctx, n_new = 24, 16
    Ca, Cb, Za, Zb = (r.normal(size=(n_ctx + n_new, c)) for _ in range(4))
    Ba, Bb = r.normal(size=(m, c)) * 0.1, r.normal(size=(m, c)) * 0.1
    whole = O.compress(Ca, Za, m, Ba, Cb, Zb, Bb)
    chunk = O.compress(Ca[n_ctx:], Za[n_ctx:], m, Ba, Cb[n_ctx:], Zb[n_ctx:], Bb,
                       prev_Cb=Cb[n_ctx - m:n_ctx], prev_Zb=Zb[n_ctx - m:n_ctx])
    np.testing.assert_allclose(chunk, whole[n_ctx // m:], rtol=1e-14, atol=1e-15)


def test_output_is_convex_combination():
    r = _rng(8)
    m, c = 4, 32
    Ca, Cb, Za, Zb = (r.normal(size=(8 * m, c)) for _ in range(4))
    y = O.compress(Ca, Za, m, None, Cb, Zb, None)
    for i in range(1, 8):
        vals = np.concatenate([Ca[m * i:m * i + m], Cb[m * i - m:m * i]])
        assert np.all(y[i] <= vals.max(0) + 1e-12) and np.all(y[i] >= vals.min(0) - 1e-12)


def test_write_epilogue_norm_and_rope():
    r = _rng(9)
    E = r.normal(size=(6, 512)) * 3
    out = O.compress_write(E, O.NORM_W | O.ROPE_W, m=2, pos0=10)
    # RMSNorm gives unit RMS; RoPE is a rotation, so the RMS stays 1
    np.testing.assert_allclose(np.sqrt(np.mean(out ** 2, axis=1)), np.ones(6), rtol=1e-6)
    # the first 448 channels are only normalised
    np.testing.assert_allclose(out[:, :448], O.rms_norm(E)[:, :448], rtol=1e-14)
    # rotating back by each entry's position (pos0 + m*i) undoes the RoPE
    for i in range(6):
        back = O.rope(out[i], 10 + 2 * i, inverse=True)
        np.testing.assert_allclose(back, O.rms_norm(E)[i], rtol=1e-12, atol=1e-12)
