"""Pins for the oracle's shared-KV attention with window, sink, RMSNorm and RoPE."""
import math

import numpy as np
import pytest

from oracle import csa2_oracle as O


def test_worked_example(golden):
    g = golden("sparse_shared_kv_example.json")
    hd = g["hand_derived"]
    kv = np.array(g["kv"])
    o, lse, mass = O.sparse_attn(np.array([g["q"]]), kv, np.array(hd["ids_ascending"]),
                                 swa=np.zeros((1, 2)), swa_pos0=0, t=0,
                                 sink=np.array([g["sink_logit"]]), window=0, flags=0)
    assert o.shape == (1, 2)
    assert 0 < mass[0] < 1
    np.testing.assert_allclose(o[0], hd["out"], rtol=1e-9)
    np.testing.assert_allclose(mass[0], hd["mass"], rtol=1e-9)
    a, b = math.exp(math.sqrt(2)), math.exp(1 / math.sqrt(2))
    np.testing.assert_allclose(lse[0], math.log(a + b + 1), rtol=1e-14)


def test_no_sink_mass_is_one_and_finite_sink_below_one():
    r = np.random.default_rng(1)
    q, K = r.normal(size=(4, 64)), r.normal(size=(30, 64))
    _, _, mass = O.attend(q, K, t=5, sink=None, flags=O.QNORM | O.KVNORM | O.ROPE)
    np.testing.assert_allclose(mass, np.ones(4), rtol=1e-14)
    _, _, mass = O.attend(q, K, t=5, sink=np.array([-1e308] * 4))
    np.testing.assert_allclose(mass, np.ones(4), rtol=1e-14)
    _, _, mass = O.attend(q, K, t=5, sink=r.normal(size=4))
    assert np.all((mass > 0) & (mass < 1))


def test_extreme_logits_stay_finite():
    q = np.zeros((2, 64))
    q[:, 0] = 1e4
    K = np.zeros((5, 64))
    K[:, 0] = np.array([1e4, -1e4, 3e3, 0, 1])
    o, lse, mass = O.attend(q, K, t=0, sink=np.array([500.0, -500.0]), flags=0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert mass[1] == pytest.approx(1.0)


def _dense_masked_reference(q, kv, swa, swa_pos0, t, V, window, sink):
    """Brute force: dense attention over ALL compressed entries and all window
    slots with an explicit mask (visible entries + window positions), written with
    loops; no RMSNorm/RoPE."""
    H, c = q.shape
    keys = []
    for s in range(kv.shape[0]):
        if s < V:
            keys.append(kv[s])
    cap = swa.shape[0]
    for p in range(0, t + 1):
        if p >= t - window + 1 and p >= 0:
            keys.append(swa[(p - swa_pos0) % cap])
    out = np.zeros((H, c))
    for h in range(H):
        z = [sum(q[h, d] * k[d] for d in range(c)) / math.sqrt(c) for k in keys]
        mx = max(z + [sink[h]])
        e = [math.exp(v - mx) for v in z]
        den = sum(e) + math.exp(sink[h] - mx)
        for j, k in enumerate(keys):
            out[h] += e[j] / den * k
    return out


def test_sparse_with_all_visible_equals_dense_masked():
    r = np.random.default_rng(2)
    H, c, N = 3, 8, 40
    q, kv = r.normal(size=(H, c)), r.normal(size=(N, c))
    swa = r.normal(size=(16, c))
    t, V, window = 21, 17, 5
    sink = r.normal(size=H)
    idx = np.concatenate([np.arange(V), -np.ones(7, dtype=int)])
    o, _, _ = O.sparse_attn(q, kv, idx, swa, 0, t, sink, window, flags=0)
    np.testing.assert_allclose(o, _dense_masked_reference(q, kv, swa, 0, t, V, window, sink),
                               rtol=1e-12, atol=1e-12)


def test_window_ring_slots_and_start():
    r = np.random.default_rng(3)
    c = 8
    swa = r.normal(size=(4, c))
    k = O.gather_keys(np.zeros((1, c)), np.array([-1]), swa, 0, t=9, window=4)
    np.testing.assert_array_equal(k, swa[[6 % 4, 7 % 4, 8 % 4, 9 % 4]])
    k = O.gather_keys(np.zeros((1, c)), np.array([-1]), swa, 0, t=1, window=4)
    np.testing.assert_array_equal(k, swa[[0, 1]])          # window clipped at position 0
    lin = r.normal(size=(10, c))                           # linear buffer from position 100
    k = O.gather_keys(np.zeros((1, c)), np.array([-1]), lin, 100, t=105, window=3)
    np.testing.assert_array_equal(k, lin[[3, 4, 5]])


def test_rms_norm_scale_invariance():
    r = np.random.default_rng(4)
    q, K = r.normal(size=(4, 512)), r.normal(size=(20, 512))
    sink = r.normal(size=4)
    o1, _, _ = O.attend(q, K, 77, sink)
    # scales in [1/4, 4]: mean(x^2) >= 1/16 stays far above the 1e-6 epsilon, whose
    # relative effect on a row's norm is then below 2e-5 (logits up to ~25 move by
    # < 5e-4, outputs by < 5e-5)
    alpha = np.exp(np.clip(r.normal(size=(20, 1)), -1.38, 1.38))
    o2, _, _ = O.attend(q * 3.7, K * alpha, 77, sink)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=5e-5)
    # without the norms the same scaling changes the result by far more
    o3, _, _ = O.attend(q * 3.7, K * alpha, 77, sink, flags=O.ROPE)
    assert np.max(np.abs(o3 - O.attend(q, K, 77, sink, flags=O.ROPE)[0])) > 1e-1


def test_rope_inverse_and_norm():
    r = np.random.default_rng(5)
    x = r.normal(size=(3, 512))
    for pos in (0, 1, 4095, 1 << 20):
        y = O.rope(x, pos)
        np.testing.assert_array_equal(y[:, :448], x[:, :448])
        np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
        np.testing.assert_allclose(O.rope(y, pos, inverse=True), x, rtol=1e-11, atol=1e-11)


def test_rope_shift_invariance_of_attention():
    # Keys are stored rotated at their own positions; the query is rotated at t and
    # the output rotated back by t.  Shifting t and every key position by the same
    # amount must leave the output unchanged: each value's contribution depends only
    # on the query-key offset (DSA-to-CSA/HCA page, §Shared-KV MQA).
    r = np.random.default_rng(6)
    H, c, n = 4, 512, 24
    q = r.normal(size=(H, c))
    raw = r.normal(size=(n, c))
    offs = r.integers(0, 5000, size=n)
    sink = r.normal(size=H)
    outs = []
    for shift in (0, 12345, 1 << 20):
        t = 6000 + shift
        stored = np.stack([O.rope(raw[j], t - offs[j]) for j in range(n)])
        o, lse, _ = O.attend(q, stored, t, sink)
        outs.append((o, lse))
    for o, lse in outs[1:]:
        np.testing.assert_allclose(o, outs[0][0], rtol=1e-7, atol=1e-9)
        np.testing.assert_allclose(lse, outs[0][1], rtol=1e-9)


def test_merge_of_partial_attention():
    r = np.random.default_rng(7)
    H, c = 4, 64
    q, K = r.normal(size=(H, c)), r.normal(size=(50, c))
    sink = r.normal(size=H)
    o_full, lse_full, _ = O.attend(q, K, 9, sink)
    parts = [O.attend(q, K[a:b], 9, None) for a, b in ((0, 13), (13, 40), (40, 50))]
    o, L = O.merge_attn([p[0] for p in parts], [p[1] for p in parts], sink)
    np.testing.assert_allclose(o, o_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, lse_full, rtol=1e-13)


def test_full_layer_decode_tiny_workload():
    # the tiny fp32 workload through the oracle end to end: shapes and invariants
    import torch
    from compressed_sparse_attention_06_gb300 import workloads as W
    wl = W.tiny_full_layer("cpu")
    E = O.compress(wl["Ca"].numpy(), wl["Za"].numpy(), wl.m, wl["Ba"].numpy())
    kv = O.compress_write(E, O.NORM_W | O.ROPE_W, wl.m, 0)
    res = O.full_layer_decode(wl["qI"][0].numpy(), wl["w"][0].numpy(), wl["KI"][0].numpy(),
                              wl["q"][0].numpy(), kv, wl["swa"][0].numpy(), 0,
                              wl.q_pos[0].numpy(), wl.m, wl["sink"].numpy())
    for i, t in enumerate(wl.q_pos[0].tolist()):
        V = t // 2
        ids = res[i]["idx"]
        assert np.all(ids >= 0) and np.all(ids < V) and len(set(ids.tolist())) == 512
        assert np.all(np.diff(ids) > 0)
        assert np.all((res[i]["mass"] > 0) & (res[i]["mass"] < 1))
        assert res[i]["out"].shape == (16, 512)


def test_hca_dense_attention_identical_rows_closed_form():
    """HCA (DSA-to-CSA/HCA page eq. 26): when every visible entry and every window row
    is the same vector x, the weights do not matter -- without a sink the output is
    the inverse rotation of the normalised row, RoPE_{-t}(x / rms(x)), for any query."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(512)
    m, t, H = 128, 128 * 9 + 40, 3
    kv = np.tile(x, (20, 1))
    swa = np.tile(x, (128, 1))
    q = rng.standard_normal((H, 512))
    out, lse, mass = O.dense_attn(q, kv, swa, 0, t, m, None, 128)
    expect = O.rope(O.rms_norm(x), t, inverse=True)
    for h in range(H):
        np.testing.assert_allclose(out[h], expect, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mass, 1.0, rtol=1e-12)


def test_hca_dense_attention_sees_exactly_the_completed_blocks():
    """Query t sees entries 0 .. floor(t/m)-1 (t >= m(j+1)): changing the first entry
    it cannot see leaves the output unchanged, changing the last one it can see
    changes it, and so does changing entry 0."""
    rng = np.random.default_rng(6)
    m, H = 128, 2
    kv = rng.standard_normal((12, 512))
    swa = rng.standard_normal((128, 512))
    q = rng.standard_normal((H, 512))
    for t in (128 * 5 - 1, 128 * 5, 128 * 5 + 77):
        V = t // m
        base, _, _ = O.dense_attn(q, kv, swa, 0, t, m)
        for j, changes in ((V, False), (V - 1, True), (0, True)):
            kv2 = kv.copy()
            kv2[j] = rng.standard_normal(512) * 3
            o2, _, _ = O.dense_attn(q, kv2, swa, 0, t, m)
            assert (np.max(np.abs(o2 - base)) > 1e-6) == changes, (t, j)
