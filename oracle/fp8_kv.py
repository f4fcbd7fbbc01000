"""CPU oracle for the FP8 (e4m3) paged KV cache with per-block scales.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
the bench's CPU-baseline / reference legs may import this module. It shares
no code with the CUDA library: numpy (float32 for the steps the format fixes
in single precision, float64 for attention) and nothing else.

Sources:
[P1] "Tech Radar: vLLM v1 Production Engine Architecture & Distributed KV
     Cache Optimization", section 2 "Memory Virtualization: PagedAttention v3
     & Hopper TMA Asynchrony", subsection "Hopper TMA Warp Specialization &
     FP8 Kernel Integration", item 3 "FP8 Block-Quantized Caching": keys and
     values are quantized dynamically to 8-bit floating point (e4m3 or e5m2)
     at block boundaries, halving the bytes per token.
[P2] "High-Throughput Local LLM Infrastructure...", section 6 "Real-World
     Developer Q&A Breakdown", Q5 (FP8 KV cache): one byte per element
     instead of two; the accuracy figure is quoted for e4m3.
The e4m3 format itself is the OCP 8-bit floating point format E4M3 (the one
the pages name "fp8_e4m3"): sign bit, 4 exponent bits with bias 7, 3 mantissa
bits; exponent field 0 encodes subnormals m * 2^-9; the all-ones pattern
S.1111.111 is NaN; there is no infinity; the largest finite magnitude is
1.75 * 2^8 = 448.

Readings where the pages are silent (each is listed in the design notes):
  * granularity: one fp32 scale per (physical block, KV head), separately for
    the K and the V pool ("at block boundaries"), stored as
    scales[block, kv_head, 0 (K) / 1 (V)];
  * stored value = decode(code) * scale; code = e4m3(x / scale) with
    round-to-nearest-even and saturation to +-448;
  * scale of a block = (largest |x| written into it) / 448, so the largest
    element uses the top code;
  * "dynamically": a write that starts a block (touches offset 0) starts it
    afresh (its old scale and codes are ignored); a write that appends to a
    block (all touched offsets > 0) keeps the old scale unless the new rows
    need a larger one, and then re-encodes the codes at offsets below the
    first touched offset (the tokens already in the block) to the new scale;
  * the arithmetic of those steps is single precision, as the format fixes
    it: s_new = fl32(amax / 448), code = e4m3(fl32(x / s)), re-encoded code =
    e4m3(fl32(decode(c) * fl32(s_old / s_new))); a scale of 0 (all rows
    zero) gives code 0;
  * e5m2, the other format [P1] names, follows the same rule with its own
    codec and largest finite value: OCP FP8 E5M2 (sign bit, 5 exponent bits
    with bias 15, 2 mantissa bits; exponent field 0 encodes subnormals
    m * 2^-16; exponent field 31 encodes infinity (m = 0) and NaN (m != 0);
    the largest finite magnitude is 1.75 * 2^15 = 57344). Encoding rounds to
    nearest even and saturates at +-57344 (an infinite input included), so
    a code written by the cache is always finite. The e5m2 functions are
    separate functions below (suffix _e5m2); the e4m3 ones are unchanged.

Pins: tests/test_oracle_fp8_pins.py checks every function here against
torch's float8_e4m3fn / float8_e5m2 dtypes, the format's closed forms, the rounding error
bound and exact invariants of the scale rule, with planted mistakes that the
pins must catch. No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


# ---------------------------------------------------------------------------
# The e4m3 format (OCP 8-bit floating point, E4M3).
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of every code as float64 (exact): (-1)^s * 2^(e-7) * (1 + m/8)
    for e > 0, (-1)^s * 2^-6 * (m/8) for e = 0, NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    val = sign * np.where(e > 0, normal, sub)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(x) -> np.ndarray:
    """Round float32 values to the nearest e4m3 code (ties to even mantissa),
    magnitudes above 448 saturate to 448, NaN gives 0x7F. Sign kept (also for
    zero and for values that round to zero)."""
    xf = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(xf)
    a = np.minimum(np.abs(xf), E4M3_MAX)
    a = np.where(np.isnan(xf), 0.0, a)
    # Exponent of the binade of a (a in [2^e, 2^(e+1))), floored at the
    # subnormal binade: the spacing of representable values there is 2^(e-3).
    _, ex = np.frexp(a)
    e = np.maximum(ex.astype(np.int64) - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    q = np.rint(a / quantum) * quantum          # a / quantum is exact; rint ties to even
    # Encode the rounded magnitude (rounding may have moved it up one binade).
    _, qe = np.frexp(q)
    qe = qe.astype(np.int64) - 1
    is_normal = q >= 2.0 ** -6
    efield = np.where(is_normal, qe + 7, 0)
    mfield = np.where(is_normal, np.rint((q / np.ldexp(1.0, qe) - 1.0) * 8.0), np.rint(q / 2.0 ** -9))
    mag = (efield << 3) | mfield.astype(np.int64)
    code = np.where(neg, 0x80, 0) | mag
    code = np.where(np.isnan(xf), E4M3_NAN, code)
    return code.astype(np.uint8)


# ---------------------------------------------------------------------------
# Cache writes with per-block scales ([P1] item 3: quantized dynamically at
# block boundaries).
# ---------------------------------------------------------------------------

def _f32(x):
    return np.float32(x)


def write_block_rows(codes: np.ndarray, scale: np.float32, offsets, rows) -> np.float32:
    """Write `rows` (float32 [n, D]) at `offsets` of one (block, KV head) tile
    of one pool: codes uint8 [B, D], updated in place. Returns the new scale.

    Steps, in order: a = largest |x| of the new rows; if the write touches
    offset 0 the block starts afresh (s_old = 0), else s_old = the stored
    scale; s_new = max(s_old, fl32(a / 448)); if s_new > s_old > 0 the codes
    at offsets below the first touched one are re-encoded with ratio
    fl32(s_old / s_new); then every new row is encoded with s_new."""
    offsets = [int(o) for o in offsets]
    rows = np.asarray(rows, dtype=np.float32).reshape(len(offsets), -1)
    o_min = min(offsets)
    with np.errstate(invalid="ignore"):
        a = _f32(np.fmax.reduce(np.abs(rows), axis=None)) if rows.size else _f32(0.0)
    s_old = _f32(0.0) if o_min == 0 else _f32(scale)
    s_new = max(s_old, _f32(a / _f32(E4M3_MAX)))
    s_new = _f32(s_new)
    if s_new > s_old and s_old > 0 and o_min > 0:
        r = _f32(s_old / s_new)
        old = e4m3_decode(codes[:o_min]).astype(np.float32)
        codes[:o_min] = e4m3_encode((old * r).astype(np.float32))
    for o, x in zip(offsets, rows):
        if s_new > 0:
            codes[o] = e4m3_encode((x / s_new).astype(np.float32))
        else:
            codes[o] = 0
    return s_new


def reshape_and_cache_fp8(k_new, v_new, slots, k_codes, v_codes, scales, block_size: int) -> None:
    """In place: the new tokens (float32 [T, Hkv, D]) go to their slots of the
    e4m3 pools (uint8 [P, Hkv, B, D]); scales float32 [P, Hkv, 2] (K, V).
    All tokens of one call that land in one block are written together (one
    write_block_rows per block, KV head and pool); slot < 0 skips a token."""
    k_new = np.asarray(k_new, dtype=np.float32)
    v_new = np.asarray(v_new, dtype=np.float32)
    by_block: dict[int, list[tuple[int, int]]] = {}
    for t, slot in enumerate(np.asarray(slots)):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        by_block.setdefault(blk, []).append((off, t))
    hkv = k_codes.shape[1]
    for blk, items in by_block.items():
        offs = [o for o, _ in items]
        toks = [t for _, t in items]
        for h in range(hkv):
            scales[blk, h, 0] = write_block_rows(k_codes[blk, h], scales[blk, h, 0], offs, k_new[toks, h])
            scales[blk, h, 1] = write_block_rows(v_codes[blk, h], scales[blk, h, 1], offs, v_new[toks, h])


def quantize_fresh_blocks(values) -> tuple[np.ndarray, np.ndarray]:
    """Codes uint8 [P, Hkv, B, D] and scales float32 [P, Hkv] of whole blocks
    written in one call each (every offset touched, so every block starts
    afresh): s = fl32(amax / 448) per (block, KV head), code = e4m3(fl32(x / s)).
    The vectorised form of write_block_rows for that case (the pins check
    that the two agree)."""
    x = np.asarray(values, dtype=np.float32)
    with np.errstate(invalid="ignore"):
        a = np.fmax.reduce(np.abs(x), axis=(2, 3)).astype(np.float32)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    codes = e4m3_encode((x / safe[:, :, None, None]).astype(np.float32))
    codes = np.where(s[:, :, None, None] > 0, codes, np.uint8(0)).astype(np.uint8)
    return codes, s


def dequantize(codes, scale_kv) -> np.ndarray:
    """Stored values of a pool as float64 [P, Hkv, B, D]: decode(code) times
    the (block, KV head) scale (exact in float64: at most 4 + 24 significant
    bits)."""
    return e4m3_decode(codes) * np.asarray(scale_kv, dtype=np.float64)[:, :, None, None]


def copy_blocks_fp8(k_codes, v_codes, scales, pairs) -> None:
    """Copy-on-write for the e4m3 pools: the whole K and V blocks and their
    scales, dst <- src, for every pair."""
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        k_codes[int(dst)] = k_codes[int(src)]
        v_codes[int(dst)] = v_codes[int(src)]
        scales[int(dst)] = scales[int(src)]


# ---------------------------------------------------------------------------
# The e5m2 format (OCP 8-bit floating point, E5M2), the other 8-bit format of
# [P1] item 3, and the same per-block cache rule with its codec.
# ---------------------------------------------------------------------------

E5M2_MAX = 57344.0
E5M2_NAN = 0x7F


def e5m2_decode(codes) -> np.ndarray:
    """Value of every code as float64 (exact): (-1)^s * 2^(e-15) * (1 + m/4)
    for 0 < e < 31, (-1)^s * 2^-14 * (m/4) for e = 0, (-1)^s * infinity for
    e = 31 with m = 0, NaN for e = 31 with m != 0."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = c & 0x3
    normal = np.ldexp(1.0 + m / 4.0, (e - 15).astype(np.int64))
    sub = np.ldexp(m / 4.0, -14)
    val = sign * np.where(e > 0, normal, sub)
    special = np.where(m == 0, sign * np.inf, np.nan)
    return np.where(e == 31, special, val)


def e5m2_encode(x) -> np.ndarray:
    """Round float32 values to the nearest e5m2 code (ties to even mantissa);
    magnitudes above 57344 (infinity included) saturate to 57344; NaN gives
    0x7F. Sign kept (also for zero and for values that round to zero)."""
    xf = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(xf)
    a = np.minimum(np.abs(xf), E5M2_MAX)
    a = np.where(np.isnan(xf), 0.0, a)
    # Binade of a (a in [2^e, 2^(e+1))), floored at the subnormal binade: the
    # spacing of representable values there is 2^(e-2).
    _, ex = np.frexp(a)
    e = np.maximum(ex.astype(np.int64) - 1, -14)
    quantum = np.ldexp(1.0, e - 2)
    q = np.rint(a / quantum) * quantum          # a / quantum is exact; rint ties to even
    _, qe = np.frexp(q)
    qe = qe.astype(np.int64) - 1
    is_normal = q >= 2.0 ** -14
    efield = np.where(is_normal, qe + 15, 0)
    mfield = np.where(is_normal, np.rint((q / np.ldexp(1.0, qe) - 1.0) * 4.0), np.rint(q / 2.0 ** -16))
    mag = (efield << 2) | mfield.astype(np.int64)
    code = np.where(neg, 0x80, 0) | mag
    code = np.where(np.isnan(xf), E5M2_NAN, code)
    return code.astype(np.uint8)


def write_block_rows_e5m2(codes: np.ndarray, scale: np.float32, offsets, rows) -> np.float32:
    """write_block_rows with the e5m2 codec: a = largest |x| of the new rows;
    s_old = 0 if the write touches offset 0, else the stored scale; s_new =
    max(s_old, fl32(a / 57344)); if s_new > s_old > 0 the codes below the
    first touched offset are re-encoded with ratio fl32(s_old / s_new); every
    new row is encoded as e5m2(fl32(x / s_new)) (code 0 when s_new == 0)."""
    offsets = [int(o) for o in offsets]
    rows = np.asarray(rows, dtype=np.float32).reshape(len(offsets), -1)
    o_min = min(offsets)
    with np.errstate(invalid="ignore"):
        a = _f32(np.fmax.reduce(np.abs(rows), axis=None)) if rows.size else _f32(0.0)
    s_old = _f32(0.0) if o_min == 0 else _f32(scale)
    s_new = _f32(max(s_old, _f32(a / _f32(E5M2_MAX))))
    if s_new > s_old and s_old > 0 and o_min > 0:
        r = _f32(s_old / s_new)
        old = e5m2_decode(codes[:o_min]).astype(np.float32)
        codes[:o_min] = e5m2_encode((old * r).astype(np.float32))
    for o, x in zip(offsets, rows):
        if s_new > 0:
            codes[o] = e5m2_encode((x / s_new).astype(np.float32))
        else:
            codes[o] = 0
    return s_new


def reshape_and_cache_e5m2(k_new, v_new, slots, k_codes, v_codes, scales, block_size: int) -> None:
    """reshape_and_cache_fp8 into e5m2 pools: one write_block_rows_e5m2 per
    (block, KV head, pool) over all the call's tokens in that block; slot < 0
    skips a token."""
    k_new = np.asarray(k_new, dtype=np.float32)
    v_new = np.asarray(v_new, dtype=np.float32)
    by_block: dict[int, list[tuple[int, int]]] = {}
    for t, slot in enumerate(np.asarray(slots)):
        slot = int(slot)
        if slot < 0:
            continue
        by_block.setdefault(slot // block_size, []).append((slot % block_size, t))
    hkv = k_codes.shape[1]
    for blk, items in by_block.items():
        offs = [o for o, _ in items]
        toks = [t for _, t in items]
        for h in range(hkv):
            scales[blk, h, 0] = write_block_rows_e5m2(k_codes[blk, h], scales[blk, h, 0], offs, k_new[toks, h])
            scales[blk, h, 1] = write_block_rows_e5m2(v_codes[blk, h], scales[blk, h, 1], offs, v_new[toks, h])


def quantize_fresh_blocks_e5m2(values) -> tuple[np.ndarray, np.ndarray]:
    """quantize_fresh_blocks with the e5m2 codec: s = fl32(amax / 57344) per
    (block, KV head), code = e5m2(fl32(x / s))."""
    x = np.asarray(values, dtype=np.float32)
    with np.errstate(invalid="ignore"):
        a = np.fmax.reduce(np.abs(x), axis=(2, 3)).astype(np.float32)
    s = (a / np.float32(E5M2_MAX)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    codes = e5m2_encode((x / safe[:, :, None, None]).astype(np.float32))
    codes = np.where(s[:, :, None, None] > 0, codes, np.uint8(0)).astype(np.uint8)
    return codes, s


def dequantize_e5m2(codes, scale_kv) -> np.ndarray:
    """Stored values of an e5m2 pool as float64 [P, Hkv, B, D]: decode(code)
    times the (block, KV head) scale (exact in float64)."""
    return e5m2_decode(codes) * np.asarray(scale_kv, dtype=np.float64)[:, :, None, None]
