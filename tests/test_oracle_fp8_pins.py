"""Pins of the FP8 (e4m3, e5m2) KV-cache oracle to things other than itself (no GPU).

What pins what:
  * torch's float8_e4m3fn dtype (a library implementation of the OCP E4M3
    format) pins the decoder on all 256 codes and the encoder (round to
    nearest, ties to even) on random values over every binade, on every
    representable value and on every midpoint between neighbours;
  * the format's closed forms: 448 is the largest finite value, values
    beyond it saturate, subnormals are m * 2^-9;
  * the quantiser's error bound: half a unit in the last place of e4m3
    (2^-4 relative in the normal range, 2^-10 * scale below it);
  * exact invariants of the per-block scale rule: a fresh block's largest
    element takes the top code and its scale is fl32(amax / 448); appending
    rows that do not need a larger scale gives the same codes as one write;
    a scale that grows by a power of two leaves every re-encoded normal
    value unchanged; a write at offset 0 forgets the old scale;
  * the vectorised whole-block quantiser equals the per-row rule;
  * copy-on-write moves codes and scales (dequantised blocks identical);
  * the e5m2 codec and rule the same way: torch's float8_e5m2 dtype on all
    256 codes and on every in-range value and tie (torch's cast overflows to
    infinity where the cache saturates, so saturation is pinned by its
    closed form), the half-ulp bound (2^-3 relative, 2^-17 * scale below the
    normal range), the top code 0x7B for a block's largest element, appends,
    the vectorised form and the cache write over several blocks.
Planted mistakes at the bottom must each fail at least one pin.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_kv as f8


def torch_encode(x) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_decode(codes) -> np.ndarray:
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _grid():
    v = torch_decode(np.arange(256, dtype=np.uint8))
    return np.unique(np.abs(v[~np.isnan(v)]))


def roundtrip_bound(x, s):
    """|decode(code) * s - x| allowed by one e4m3 rounding of x / s (plus the
    fp32 division's own rounding)."""
    return (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s) * (1 + 2.0 ** -20)


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------

def pin_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_decode(codes)
    got = f8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    # Closed forms of the format.
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x38] == 1.0


def pin_encode_vs_torch():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(100_000) * np.exp2(rng.uniform(-14, 9, 100_000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    g = _grid()
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)        # exact ties: round half to even
    x = np.concatenate([x, g.astype(np.float32), -g.astype(np.float32), mids, -mids,
                        np.float32([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, 3 * 2.0 ** -11])])
    assert np.array_equal(f8.e4m3_encode(x), torch_encode(x))


def pin_encode_saturates():
    got = f8.e4m3_encode(np.float32([448, 449, 463.9, 464, 1000, np.inf, -470, -np.inf]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(f8.e4m3_encode(f8.e4m3_decode(codes).astype(np.float32)), codes)


def _rows(rng, n, d, mag=1.0):
    return (rng.standard_normal((n, d)) * mag).astype(np.float32)


def pin_fresh_block():
    rng = np.random.default_rng(12)
    for mag in (1.0, 1e-3, 37.0, 1e-6):
        x = _rows(rng, 16, 64, mag)
        codes = np.zeros((16, 64), np.uint8)
        s = f8.write_block_rows(codes, np.float32(5.0), range(16), x)
        a = np.float32(np.abs(x).max())
        assert s == np.float32(a / np.float32(448.0))
        i = np.unravel_index(np.abs(x).argmax(), x.shape)
        assert codes[i] in (0x7E, 0xFE)
        err = np.abs(torch_decode(codes) * np.float64(s) - x)
        assert (err <= roundtrip_bound(x, s)).all()
    # All-zero rows: scale 0, codes 0, values 0.
    codes = np.full((16, 64), 0x55, np.uint8)
    s = f8.write_block_rows(codes, np.float32(1.0), range(16), np.zeros((16, 64), np.float32))
    assert s == 0 and (codes == 0).all()


def pin_append_without_growth():
    rng = np.random.default_rng(13)
    x = _rows(rng, 32, 128)
    x[3, 7] = 9.0                                           # the block's maximum comes first
    one = np.zeros((32, 128), np.uint8)
    s_one = f8.write_block_rows(one, np.float32(0), range(32), x)
    two = np.zeros((32, 128), np.uint8)
    s = f8.write_block_rows(two, np.float32(0), range(10), x[:10])
    s = f8.write_block_rows(two, s, range(10, 11), x[10:11])
    s = f8.write_block_rows(two, s, range(11, 32), x[11:])
    assert s == s_one and np.array_equal(one, two)


def pin_append_with_growth():
    rng = np.random.default_rng(14)
    # Old rows: every value in the normal range even after the scale grows 4x
    # (|x / s| >= 2^-4 before, >= 2^-6 after), so re-encoding by the exact
    # ratio 1/4 changes no value.
    base = rng.uniform(0.5, 1.0, (8, 64)) * rng.choice([-1, 1], (8, 64))
    base[0, 0] = 1.0
    old = base.astype(np.float32)
    codes = np.zeros((16, 64), np.uint8)
    s0 = f8.write_block_rows(codes, np.float32(0), range(8), old)
    before = torch_decode(codes[:8]) * np.float64(s0)
    new = np.zeros((2, 64), np.float32)
    new[1, 5] = 4.0                                         # amax grows exactly 4x
    s1 = f8.write_block_rows(codes, s0, [8, 9], new)
    assert s1 == np.float32(4.0 / np.float32(448.0)) and s1 == 4 * s0
    after = torch_decode(codes[:8]) * np.float64(s1)
    assert np.array_equal(before, after)
    # A growth by a non-power-of-two keeps every old value within two roundings.
    codes2 = np.zeros((16, 64), np.uint8)
    x = _rows(rng, 8, 64)
    t0 = f8.write_block_rows(codes2, np.float32(0), range(8), x)
    t1 = f8.write_block_rows(codes2, t0, [8], _rows(rng, 1, 64, 7.3))
    assert t1 > t0
    err = np.abs(torch_decode(codes2[:8]) * np.float64(t1) - x)
    xhat = torch_decode(f8.e4m3_encode((x / t0).astype(np.float32))) * np.float64(t0)
    assert (err <= roundtrip_bound(x, t0) + roundtrip_bound(xhat, t1)).all()
    # Offsets above the write are not touched.
    codes3 = np.full((16, 64), 0x33, np.uint8)
    f8.write_block_rows(codes3, np.float32(0), range(4), _rows(rng, 4, 64))
    assert (codes3[4:] == 0x33).all()


def pin_fresh_write_forgets_old_scale():
    rng = np.random.default_rng(15)
    codes = np.zeros((16, 64), np.uint8)
    s = f8.write_block_rows(codes, np.float32(0), range(16), _rows(rng, 16, 64, 100.0))
    small = _rows(rng, 1, 64, 0.01)
    s2 = f8.write_block_rows(codes, s, [0], small)
    assert s2 == np.float32(np.float32(np.abs(small).max()) / np.float32(448.0))


def pin_fresh_blocks_vectorised():
    rng = np.random.default_rng(16)
    vals = (rng.standard_normal((5, 3, 16, 32)) * np.exp2(rng.uniform(-8, 4, (5, 3, 1, 1)))).astype(np.float32)
    vals[2, 1] = 0.0
    codes, scales = f8.quantize_fresh_blocks(vals)
    for b in range(5):
        for h in range(3):
            c = np.zeros((16, 32), np.uint8)
            s = f8.write_block_rows(c, np.float32(0), range(16), vals[b, h])
            assert s == scales[b, h] and np.array_equal(c, codes[b, h])


def pin_reshape_and_cache_fp8():
    rng = np.random.default_rng(17)
    P, H, B, D = 6, 2, 16, 32
    kc = np.zeros((P, H, B, D), np.uint8)
    vc = np.zeros((P, H, B, D), np.uint8)
    sc = np.zeros((P, H, 2), np.float32)
    # Block 4 gets offsets 0..9 of one sequence, block 1 offsets 0..2 of
    # another, one padding token.
    slots = np.array([4 * B + o for o in range(10)] + [-1] + [1 * B + o for o in range(3)])
    k = _rows(rng, len(slots) * H, D).reshape(len(slots), H, D)
    v = _rows(rng, len(slots) * H, D, 3.0).reshape(len(slots), H, D)
    f8.reshape_and_cache_fp8(k, v, slots, kc, vc, sc, B)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = slot // B, slot % B
        for h in range(H):
            for pool, new, j in ((kc, k, 0), (vc, v, 1)):
                got = torch_decode(pool[blk, h, off]) * np.float64(sc[blk, h, j])
                assert (np.abs(got - new[t, h]) <= roundtrip_bound(new[t, h], sc[blk, h, j])).all()
    untouched = [0, 2, 3, 5]
    assert (kc[untouched] == 0).all() and (vc[untouched] == 0).all() and (sc[untouched] == 0).all()
    # Scales: per (block, head, pool), the largest |x| written there / 448.
    for blk, toks in ((4, range(10)), (1, range(11, 14))):
        toks = list(toks)
        for h in range(H):
            assert sc[blk, h, 0] == np.float32(np.float32(np.abs(k[toks, h]).max()) / np.float32(448))
            assert sc[blk, h, 1] == np.float32(np.float32(np.abs(v[toks, h]).max()) / np.float32(448))


def pin_dequantize_and_copy():
    rng = np.random.default_rng(18)
    vals = _rows(rng, 4 * 2 * 16, 32).reshape(4, 2, 16, 32)
    kc, ks = f8.quantize_fresh_blocks(vals)
    vc, vs = f8.quantize_fresh_blocks(vals * 2)
    scales = np.stack([ks, vs], axis=-1)
    ref = torch_decode(kc) * ks.astype(np.float64)[:, :, None, None]
    assert np.array_equal(f8.dequantize(kc, scales[..., 0]), ref)
    f8.copy_blocks_fp8(kc, vc, scales, [[0, 3], [1, 2]])
    for s, d in ((0, 3), (1, 2)):
        assert np.array_equal(f8.dequantize(kc, scales[..., 0])[d], f8.dequantize(kc, scales[..., 0])[s])
        assert np.array_equal(f8.dequantize(vc, scales[..., 1])[d], f8.dequantize(vc, scales[..., 1])[s])
    assert np.array_equal(scales[3], scales[0])


# ---------------------------------------------------------------------------
# e5m2
# ---------------------------------------------------------------------------

def torch_encode_e5m2(x) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()


def torch_decode_e5m2(codes) -> np.ndarray:
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e5m2).to(torch.float64).numpy()


def _grid_e5m2():
    v = torch_decode_e5m2(np.arange(256, dtype=np.uint8))
    return np.unique(np.abs(v[np.isfinite(v)]))


def roundtrip_bound_e5m2(x, s):
    """|decode(code) * s - x| allowed by one e5m2 rounding of x / s (plus the
    fp32 division's own rounding)."""
    return (2.0 ** -3 * np.abs(x) + 2.0 ** -17 * s) * (1 + 2.0 ** -20)


def pin_e5m2_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_decode_e5m2(codes)
    got = f8.e5m2_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    assert got[0x7B] == 57344.0 and got[0xFB] == -57344.0
    assert got[0x7C] == np.inf and got[0xFC] == -np.inf
    assert got[0x01] == 2.0 ** -16 and got[0x04] == 2.0 ** -14 and got[0x3C] == 1.0


def pin_e5m2_encode_vs_torch():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(100_000) * np.exp2(rng.uniform(-20, 16, 100_000))).astype(np.float32)
    x = x[np.abs(x) <= 57344]
    g = _grid_e5m2()
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)        # exact ties: round half to even
    x = np.concatenate([x, g.astype(np.float32), -g.astype(np.float32), mids, -mids,
                        np.float32([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -17, 3 * 2.0 ** -18, 57000.0])])
    assert np.array_equal(f8.e5m2_encode(x), torch_encode_e5m2(x))


def pin_e5m2_encode_saturates():
    got = f8.e5m2_encode(np.float32([57344, 57345, 61439, 61440, 1e9, np.inf, -70000, -np.inf]))
    assert list(got) == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0xFB]
    assert f8.e5m2_encode(np.float32([np.nan]))[0] == 0x7F
    codes = np.array([c for c in range(256) if ((c >> 2) & 0x1F) != 31], dtype=np.uint8)
    assert np.array_equal(f8.e5m2_encode(f8.e5m2_decode(codes).astype(np.float32)), codes)


def pin_e5m2_fresh_block():
    rng = np.random.default_rng(22)
    for mag in (1.0, 1e-3, 37.0, 1e-6):
        x = _rows(rng, 16, 64, mag)
        codes = np.zeros((16, 64), np.uint8)
        s = f8.write_block_rows_e5m2(codes, np.float32(5.0), range(16), x)
        a = np.float32(np.abs(x).max())
        assert s == np.float32(a / np.float32(57344.0))
        i = np.unravel_index(np.abs(x).argmax(), x.shape)
        assert codes[i] in (0x7B, 0xFB)
        err = np.abs(torch_decode_e5m2(codes) * np.float64(s) - x)
        assert (err <= roundtrip_bound_e5m2(x, s)).all()
    codes = np.full((16, 64), 0x55, np.uint8)
    s = f8.write_block_rows_e5m2(codes, np.float32(1.0), range(16), np.zeros((16, 64), np.float32))
    assert s == 0 and (codes == 0).all()


def pin_e5m2_appends():
    rng = np.random.default_rng(23)
    x = _rows(rng, 32, 128)
    x[3, 7] = 9.0
    one = np.zeros((32, 128), np.uint8)
    s_one = f8.write_block_rows_e5m2(one, np.float32(0), range(32), x)
    two = np.zeros((32, 128), np.uint8)
    s = f8.write_block_rows_e5m2(two, np.float32(0), range(10), x[:10])
    s = f8.write_block_rows_e5m2(two, s, range(10, 32), x[10:])
    assert s == s_one and np.array_equal(one, two)
    # A growth by exactly 4x leaves every re-encoded normal value unchanged.
    base = (rng.uniform(0.5, 1.0, (8, 64)) * rng.choice([-1, 1], (8, 64))).astype(np.float32)
    base[0, 0] = 1.0
    codes = np.zeros((16, 64), np.uint8)
    s0 = f8.write_block_rows_e5m2(codes, np.float32(0), range(8), base)
    before = torch_decode_e5m2(codes[:8]) * np.float64(s0)
    new = np.zeros((2, 64), np.float32)
    new[1, 5] = 4.0
    s1 = f8.write_block_rows_e5m2(codes, s0, [8, 9], new)
    assert s1 == 4 * s0
    assert np.array_equal(before, torch_decode_e5m2(codes[:8]) * np.float64(s1))
    # Any growth keeps the old values within two roundings.
    codes2 = np.zeros((16, 64), np.uint8)
    y = _rows(rng, 8, 64)
    t0 = f8.write_block_rows_e5m2(codes2, np.float32(0), range(8), y)
    t1 = f8.write_block_rows_e5m2(codes2, t0, [8], _rows(rng, 1, 64, 7.3))
    assert t1 > t0
    err = np.abs(torch_decode_e5m2(codes2[:8]) * np.float64(t1) - y)
    yhat = torch_decode_e5m2(f8.e5m2_encode((y / t0).astype(np.float32))) * np.float64(t0)
    assert (err <= roundtrip_bound_e5m2(y, t0) + roundtrip_bound_e5m2(yhat, t1)).all()


def pin_e5m2_vectorised_and_cache_write():
    rng = np.random.default_rng(24)
    vals = (rng.standard_normal((5, 3, 16, 32)) * np.exp2(rng.uniform(-8, 4, (5, 3, 1, 1)))).astype(np.float32)
    vals[2, 1] = 0.0
    codes, scales = f8.quantize_fresh_blocks_e5m2(vals)
    for b in range(5):
        for h in range(3):
            c = np.zeros((16, 32), np.uint8)
            s = f8.write_block_rows_e5m2(c, np.float32(0), range(16), vals[b, h])
            assert s == scales[b, h] and np.array_equal(c, codes[b, h])
    ref = torch_decode_e5m2(codes) * scales.astype(np.float64)[:, :, None, None]
    assert np.array_equal(f8.dequantize_e5m2(codes, scales), ref)
    P, H, B, D = 6, 2, 16, 32
    kc = np.zeros((P, H, B, D), np.uint8)
    vc = np.zeros((P, H, B, D), np.uint8)
    sc = np.zeros((P, H, 2), np.float32)
    slots = np.array([4 * B + o for o in range(10)] + [-1] + [1 * B + o for o in range(3)])
    k = _rows(rng, len(slots) * H, D).reshape(len(slots), H, D)
    v = _rows(rng, len(slots) * H, D, 3.0).reshape(len(slots), H, D)
    f8.reshape_and_cache_e5m2(k, v, slots, kc, vc, sc, B)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = slot // B, slot % B
        for h in range(H):
            for pool, new, j in ((kc, k, 0), (vc, v, 1)):
                got = torch_decode_e5m2(pool[blk, h, off]) * np.float64(sc[blk, h, j])
                assert (np.abs(got - new[t, h]) <= roundtrip_bound_e5m2(new[t, h], sc[blk, h, j])).all()
    untouched = [0, 2, 3, 5]
    assert (kc[untouched] == 0).all() and (vc[untouched] == 0).all() and (sc[untouched] == 0).all()
    for blk, toks in ((4, list(range(10))), (1, list(range(11, 14)))):
        for h in range(H):
            assert sc[blk, h, 0] == np.float32(np.float32(np.abs(k[toks, h]).max()) / np.float32(57344))
            assert sc[blk, h, 1] == np.float32(np.float32(np.abs(v[toks, h]).max()) / np.float32(57344))


ALL_PINS = [
    pin_decode_all_codes, pin_encode_vs_torch, pin_encode_saturates, pin_fresh_block,
    pin_append_without_growth, pin_append_with_growth, pin_fresh_write_forgets_old_scale,
    pin_fresh_blocks_vectorised, pin_reshape_and_cache_fp8, pin_dequantize_and_copy,
    pin_e5m2_decode_all_codes, pin_e5m2_encode_vs_torch, pin_e5m2_encode_saturates, pin_e5m2_fresh_block,
    pin_e5m2_appends, pin_e5m2_vectorised_and_cache_write,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin.
# ---------------------------------------------------------------------------

def _mut_round_half_away(monkeypatch):
    orig = f8.e4m3_encode

    def bad(x):
        xf = np.asarray(x, dtype=np.float32)
        # One fp32 ulp away from zero first: exact ties then round away from zero.
        up = np.nextafter(np.abs(xf), np.float32(np.inf)).astype(np.float32) * np.sign(xf)
        return orig(up.astype(np.float32))
    monkeypatch.setattr(f8, "e4m3_encode", bad)


def _mut_subnormal_scale(monkeypatch):
    orig = f8.e4m3_decode

    def bad(c):
        v = orig(c)
        e = (np.asarray(c, dtype=np.uint8) >> 3) & 0xF
        return np.where(e == 0, v / 2, v)
    monkeypatch.setattr(f8, "e4m3_decode", bad)


def _mut_bias8(monkeypatch):
    orig = f8.e4m3_decode
    monkeypatch.setattr(f8, "e4m3_decode", lambda c: orig(c) / 2)


def _mut_no_reencode(monkeypatch):
    def bad(codes, scale, offsets, rows):
        offsets = [int(o) for o in offsets]
        rows = np.asarray(rows, dtype=np.float32).reshape(len(offsets), -1)
        s_old = np.float32(0) if min(offsets) == 0 else np.float32(scale)
        s_new = np.float32(max(s_old, np.float32(np.abs(rows).max() / np.float32(448))))
        for o, x in zip(offsets, rows):
            codes[o] = f8.e4m3_encode((x / s_new).astype(np.float32)) if s_new > 0 else 0
        return s_new
    monkeypatch.setattr(f8, "write_block_rows", bad)


def _mut_old_scale_for_new_rows(monkeypatch):
    def bad(codes, scale, offsets, rows):
        offsets = [int(o) for o in offsets]
        rows = np.asarray(rows, dtype=np.float32).reshape(len(offsets), -1)
        s_old = np.float32(0) if min(offsets) == 0 else np.float32(scale)
        s_new = np.float32(max(s_old, np.float32(np.abs(rows).max() / np.float32(448))))
        use = s_old if s_old > 0 else s_new
        for o, x in zip(offsets, rows):
            codes[o] = f8.e4m3_encode((x / use).astype(np.float32)) if use > 0 else 0
        return s_new
    monkeypatch.setattr(f8, "write_block_rows", bad)


def _mut_keep_old_scale_when_fresh(monkeypatch):
    orig = f8.write_block_rows

    def bad(codes, scale, offsets, rows):
        offsets = list(offsets)
        if min(offsets) == 0 and scale > 0:
            rows = np.asarray(rows, dtype=np.float32).reshape(len(offsets), -1)
            s = np.float32(max(np.float32(scale), np.float32(np.abs(rows).max() / np.float32(448))))
            for o, x in zip(offsets, rows):
                codes[o] = f8.e4m3_encode((x / s).astype(np.float32))
            return s
        return orig(codes, scale, offsets, rows)
    monkeypatch.setattr(f8, "write_block_rows", bad)


def _mut_wrong_max(monkeypatch):
    monkeypatch.setattr(f8, "E4M3_MAX", 240.0)


def _mut_copy_codes_only(monkeypatch):
    def bad(kc, vc, scales, pairs):
        for s, d in np.asarray(pairs).reshape(-1, 2):
            kc[int(d)] = kc[int(s)]
            vc[int(d)] = vc[int(s)]
    monkeypatch.setattr(f8, "copy_blocks_fp8", bad)


def _mut_scale_per_block_not_head(monkeypatch):
    def bad(values):
        x = np.asarray(values, dtype=np.float32)
        a = np.abs(x).max(axis=(1, 2, 3), keepdims=True).astype(np.float32)
        s = np.broadcast_to(a / np.float32(448), x.shape[:2] + (1, 1)).astype(np.float32)
        codes = f8.e4m3_encode((x / np.where(s > 0, s, 1)).astype(np.float32))
        return codes, s[:, :, 0, 0].copy()
    monkeypatch.setattr(f8, "quantize_fresh_blocks", bad)


def _mut_e5m2_round_half_away(monkeypatch):
    orig = f8.e5m2_encode

    def bad(x):
        xf = np.asarray(x, dtype=np.float32)
        up = np.nextafter(np.abs(xf), np.float32(np.inf)).astype(np.float32) * np.sign(xf)
        return orig(up.astype(np.float32))
    monkeypatch.setattr(f8, "e5m2_encode", bad)


def _mut_e5m2_subnormal_scale(monkeypatch):
    orig = f8.e5m2_decode

    def bad(c):
        v = orig(c)
        e = (np.asarray(c, dtype=np.uint8) >> 2) & 0x1F
        return np.where(e == 0, v * 2, v)
    monkeypatch.setattr(f8, "e5m2_decode", bad)


def _mut_e5m2_bias16(monkeypatch):
    orig = f8.e5m2_decode
    monkeypatch.setattr(f8, "e5m2_decode", lambda c: orig(c) / 2)


def _mut_e5m2_e4m3_max(monkeypatch):
    monkeypatch.setattr(f8, "E5M2_MAX", 448.0)


def _mut_e5m2_no_saturation(monkeypatch):
    orig = f8.e5m2_encode

    def bad(x):
        xf = np.asarray(x, dtype=np.float32)
        c = orig(xf)
        return np.where(np.abs(xf) > 57344, np.where(np.signbit(xf), 0xFC, 0x7C), c).astype(np.uint8)
    monkeypatch.setattr(f8, "e5m2_encode", bad)


def _mut_e5m2_no_reencode(monkeypatch):
    def bad(codes, scale, offsets, rows):
        offsets = [int(o) for o in offsets]
        rows = np.asarray(rows, dtype=np.float32).reshape(len(offsets), -1)
        s_old = np.float32(0) if min(offsets) == 0 else np.float32(scale)
        s_new = np.float32(max(s_old, np.float32(np.abs(rows).max() / np.float32(57344))))
        for o, x in zip(offsets, rows):
            codes[o] = f8.e5m2_encode((x / s_new).astype(np.float32)) if s_new > 0 else 0
        return s_new
    monkeypatch.setattr(f8, "write_block_rows_e5m2", bad)


def _mut_e5m2_mantissa3(monkeypatch):
    # The e4m3 codec's grid (3 mantissa bits) behind the e5m2 names.
    monkeypatch.setattr(f8, "e5m2_encode", lambda x: f8.e4m3_encode(np.asarray(x, np.float32) / 128))


MUTATIONS = [
    _mut_round_half_away, _mut_subnormal_scale, _mut_bias8, _mut_no_reencode, _mut_old_scale_for_new_rows,
    _mut_keep_old_scale_when_fresh, _mut_wrong_max, _mut_copy_codes_only, _mut_scale_per_block_not_head,
    _mut_e5m2_round_half_away, _mut_e5m2_subnormal_scale, _mut_e5m2_bias16, _mut_e5m2_e4m3_max,
    _mut_e5m2_no_saturation, _mut_e5m2_no_reencode, _mut_e5m2_mantissa3,
]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutation, monkeypatch):
    mutation(monkeypatch)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutation.__name__}"
