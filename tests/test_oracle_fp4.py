"""Pins for the oracle's FP4 formats: the OCP code tables, RNE ties, torch's own
float8_e4m3fn conversion, brute-force nearest-value search, round trips and the
890 bytes-per-token arithmetic."""
import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O


def test_e2m1_table(golden):
    g = golden("fp4_code_tables.json")
    vals = O.e2m1_decode(np.arange(16))
    exp = np.array(g["e2m1_values_by_code"])
    np.testing.assert_array_equal(vals, exp)
    np.testing.assert_array_equal(np.signbit(vals), np.signbit(exp))


def test_e4m3_and_e8m0_selected(golden):
    g = golden("fp4_code_tables.json")
    for k, v in g["e4m3_selected"].items():
        assert O.e4m3_decode(int(k, 16)) == v, k
    for k, v in g["e8m0_selected"].items():
        assert O.e8m0_decode(int(k)) == v, k
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))
    assert np.isnan(O.e8m0_decode(255))


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(np.arange(256))
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_encode_matches_torch_in_range():
    r = np.random.default_rng(1)
    x = np.concatenate([
        r.uniform(-448, 448, 20000),
        r.normal(size=20000) * 1e-2,
        np.ldexp(r.uniform(-1, 1, 5000), r.integers(-12, 8, 5000)),
    ]).astype(np.float32)
    # every halfway point between adjacent finite codes (ties-to-even check)
    grid = O.e4m3_decode(np.arange(0x7F))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(x)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_saturates():
    assert O.e4m3_encode(1e6) == 0x7E and O.e4m3_encode(-500.0) == 0xFE
    assert O.e4m3_encode(464.0) == 0x7E


def test_e2m1_rne_ties_and_saturation(golden):
    g = golden("fp4_code_tables.json")
    for k, v in g["e2m1_rne_ties"].items():
        if k == "note":
            continue
        assert O.e2m1_decode(O.e2m1_encode(float(k))) == v, k
        assert O.e2m1_decode(O.e2m1_encode(-float(k))) == -v, k
    for k, v in g["e2m1_saturation"].items():
        assert O.e2m1_decode(O.e2m1_encode(float(k))) == v, k


def test_e2m1_sign_kept_on_zero():
    assert O.e2m1_encode(-0.1) == 0x8
    assert O.e2m1_encode(0.1) == 0x0
    assert O.e2m1_encode(-0.0) == 0x8


def test_e2m1_encode_brute_force():
    # nearest of the 8 magnitudes by exhaustive search; ties -> even code
    r = np.random.default_rng(2)
    x = np.concatenate([r.uniform(-7, 7, 50000), np.arange(-700, 701) / 100.0])
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    got = O.e2m1_encode(x)
    for xi, ci in zip(x, got):
        a = min(abs(xi), 6.0)
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert (ci & 7) == code, (xi, ci)
        assert (ci >> 3) == (1 if np.signbit(xi) else 0)


def test_row_bytes(golden):
    g = golden("cache_bytes_per_token.json")
    assert O.nvfp4_row_bytes(512) == g["main_kv_entry_bytes"] == 288
    assert O.mxfp4_row_bytes(128) == g["indexer_k_entry_bytes"] == 68
    total = 0
    for row in g["layers"]:
        per = O.nvfp4_row_bytes(512) // row["m"] + O.mxfp4_row_bytes(128) // row["m"]
        assert O.nvfp4_row_bytes(512) // row["m"] == row["main_per_token"]
        assert O.mxfp4_row_bytes(128) // row["m"] == row["index_per_token"]
        assert per * row["count"] == row["subtotal"]
        total += per * row["count"]
    assert total == g["total_bytes_per_token"] == 890


def _exact_nvfp4_rows(r, rows, c=512):
    """Rows whose values lie exactly on an FP4 grid with a scale s (an E4M3 value)
    such that each 16-group contains +-6*s, so amax/6 = s exactly."""
    codes = r.integers(0, 16, size=(rows, c))
    codes[:, ::16] = np.where(r.integers(0, 2, size=(rows, c // 16)) == 1, 0x7, 0xF)
    s_codes = r.integers(0x20, 0x50, size=(rows, c // 16))
    s = O.e4m3_decode(s_codes)
    return O.e2m1_decode(codes) * np.repeat(s, 16, axis=1), codes, s_codes


def test_nvfp4_round_trip_exact():
    r = np.random.default_rng(3)
    x, codes, s_codes = _exact_nvfp4_rows(r, 64)
    b = O.nvfp4_pack(x)
    assert b.shape == (64, 288)
    np.testing.assert_array_equal(b[:, 256:], s_codes.astype(np.uint8))
    y = O.nvfp4_unpack(b)
    np.testing.assert_array_equal(y, x)
    # nibble order: channel 2i in the low nibble of byte i
    assert (b[0, 0] & 0xF) == (O.e2m1_encode(x[0, 0] / O.e4m3_decode(s_codes[0, 0])) & 0xF)


def test_nvfp4_error_bound_and_zero_group():
    r = np.random.default_rng(4)
    x = (r.normal(size=(32, 512)) * np.exp(0.5 * r.normal(size=(32, 1)))).astype(np.float32)
    x[3, 16:32] = 0.0
    x[5, 32:48] = 1e-5   # amax/6 below the smallest E4M3 subnormal -> s = 0
    b = O.nvfp4_pack(x)
    y = O.nvfp4_unpack(b)
    assert np.all(y[3, 16:32] == 0) and np.all(b[3, 8:16] == 0) and b[3, 256 + 1] == 0
    assert np.all(y[5, 32:48] == 0) and b[5, 256 + 2] == 0
    g = x.reshape(32, 32, 16).astype(np.float64)
    s = O.e4m3_decode(b[:, 256:])
    err = np.abs(y.reshape(32, 32, 16) - g)
    # half a step of the coarsest E2M1 spacing (2 between 4 and 6) times s, plus
    # what saturation at 6*s can cost when s rounded down
    bound = s[:, :, None] * 1.0 + np.maximum(np.abs(g).max(2, keepdims=True) - 6 * s[:, :, None], 0)
    assert np.all(err <= bound + 1e-12)


def test_mxfp4_scale_rule_and_round_trip():
    r = np.random.default_rng(5)
    x = (r.normal(size=(16, 128)) * np.exp(0.5 * r.normal(size=(16, 1)))).astype(np.float32)
    x[2, 32:64] = 0.0
    b = O.mxfp4_pack(x)
    assert b.shape == (16, 68)
    amax = np.abs(x.reshape(16, 4, 32)).max(2)
    for i in range(16):
        for j in range(4):
            if amax[i, j] == 0:
                assert b[i, 64 + j] == 0 and np.all(b[i, 16 * j:16 * j + 16] == 0)
                continue
            e = int(np.floor(np.log2(amax[i, j])))
            assert b[i, 64 + j] == e - 2 + 127
            # the largest element maps into [4, 8): code 6 (value 4) or 7 (value 6)
    y = O.mxfp4_unpack(b)
    # exact representable input survives
    codes = r.integers(0, 16, size=(8, 128))
    codes[:, ::32] = 0x7                                  # group max is 6 * X
    X = np.ldexp(1.0, r.integers(-6, 4, size=(8, 4)))
    xe = O.e2m1_decode(codes) * np.repeat(X, 32, axis=1)
    np.testing.assert_array_equal(O.mxfp4_unpack(O.mxfp4_pack(xe)), xe)
    assert np.all(np.abs(y - x) <= np.repeat(O.e8m0_decode(b[:, 64:]), 32, axis=1) * 2 + 1e-12)
