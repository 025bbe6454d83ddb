"""Pins of the fp8 (E4M3) KV-cache oracle (`oracle/fp8.py`) to facts outside
itself: the bit-field definition of the format, its largest and smallest
values, round trips, ties to even, saturation, a library cast (torch's
float8_e4m3fn), per-element brute force of the quantizing append, and closed
forms of attention over a quantized cache. Planted mistakes in copies of the
oracle must each fail one of them. CPU only."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import fp8 as f8

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


# ---------------------------------------------------------------- format ---
def check_table_facts(decode):
    v = decode(np.arange(256))
    assert v[0x00] == 0.0 and not np.signbit(v[0x00])
    assert v[0x80] == 0.0 and np.signbit(v[0x80])
    assert v[0x01] == 2.0 ** -9            # smallest subnormal: 1/8 * 2^-6
    assert v[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert v[0x08] == 2.0 ** -6            # smallest normal
    assert v[0x38] == 1.0                  # exponent field 7 = bias
    assert v[0x7E] == 448.0                # 1.75 * 2^8, the largest finite
    assert v[0xFE] == -448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(v[FINITE]).all()
    mags = v[:0x7F]
    assert (np.diff(mags) > 0).all()       # codes order like their values


def check_roundtrip(encode, decode):
    c = np.array(FINITE)
    got = encode(decode(c).astype(np.float32))
    assert (got == c).all()


def check_ties_to_even(encode, decode):
    for c in range(0x7E):
        lo, hi = decode(c)[()], decode(c + 1)[()]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2              # exact in fp32
        even = c if c % 2 == 0 else c + 1
        assert encode(mid)[()] == even, c
        assert encode(np.nextafter(mid, np.float32(np.inf)))[()] == c + 1, c
        assert encode(np.nextafter(mid, np.float32(0)))[()] == c, c
        assert encode(-mid)[()] == (even | 0x80), c


def check_saturation(encode):
    assert encode(np.float32(448.0))[()] == 0x7E
    assert encode(np.float32(464.0))[()] == 0x7E         # would round to 480: saturates
    assert encode(np.float32(1e30))[()] == 0x7E
    assert encode(np.float32(-1e30))[()] == 0xFE
    assert encode(np.float32(np.inf))[()] == 0x7E
    assert encode(np.float32(-np.inf))[()] == 0xFE
    assert (encode(np.float32(np.nan))[()] & 0x7F) == 0x7F


def test_table_facts():
    check_table_facts(oracle.e4m3_decode)


def test_roundtrip_every_finite_code():
    check_roundtrip(oracle.e4m3_encode, oracle.e4m3_decode)


def test_ties_to_even():
    check_ties_to_even(oracle.e4m3_encode, oracle.e4m3_decode)


def test_saturation_and_nan():
    check_saturation(oracle.e4m3_encode)


def test_matches_torch_float8_cast():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1, 4000),
                        rng.uniform(-2.0 ** -6, 2.0 ** -6, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (oracle.e4m3_encode(x) == ref).all()


# -------------------------------------------------------------- quantize ---
def test_quantize_divides_in_fp32():
    """fp16 0x1DFD over the fp32 scale with bits 1038294130: the fp32 quotient
    is exactly the midpoint of codes 21 and 22, so the even code 22 wins; the
    exact quotient lies just below that midpoint (a wider division would give
    21). The decision is taken in fp32, the kernel's precision."""
    x = np.array([0x1DFD], dtype=np.uint16).view(np.float16)
    s = np.array([1038294130], dtype=np.uint32).view(np.float32)
    q32 = np.float32(x[0]) / s[0]
    mid = (oracle.e4m3_decode(21)[()] + oracle.e4m3_decode(22)[()]) / 2
    assert float(q32) == mid
    assert Fraction(float(np.float32(x[0]))) / Fraction(float(s[0])) < Fraction(mid)
    got = oracle.quantize_rows(x.reshape(1, 1, 1), s)
    assert got.reshape(-1)[0] == 22


def _brute_quantize(x16, scale):
    """Per element: fp32 division, then the nearest E4M3 value by scanning all
    finite codes (ties to the even code), saturating at 448."""
    vals = [(c, float(oracle.e4m3_decode(c))) for c in FINITE]
    out = np.empty(x16.shape, dtype=np.uint8)
    for idx in np.ndindex(x16.shape):
        y = float(np.float32(np.float32(x16[idx]) / np.float32(scale[idx[-2]])))
        y = max(-448.0, min(448.0, y))
        best = None
        for c, v in vals:
            if v == 0.0 and (np.signbit(v) != np.signbit(y)):
                continue
            d = abs(v - y)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
                best = (d, c)
        out[idx] = best[1]
    return out


def check_append(append):
    rng = np.random.default_rng(11)
    NB, BS, H, D = 6, 4, 2, 8
    kp = rng.integers(0, 256, (NB, BS, H, D), dtype=np.uint8)
    vp = rng.integers(0, 256, (NB, BS, H, D), dtype=np.uint8)
    kn = (rng.standard_normal((3, H, D)) * 2).astype(np.float16)
    vn = (rng.standard_normal((3, H, D)) * 2).astype(np.float16)
    ks = np.array([0.01, 0.05], dtype=np.float32)
    vs = np.array([0.03, 0.002], dtype=np.float32)
    slots = [5, -1, 17]
    k2, v2 = append(kp, vp, kn, vn, slots, ks, vs)
    ek, ev = kp.copy(), vp.copy()
    ek[1, 1] = _brute_quantize(kn[0], ks)
    ev[1, 1] = _brute_quantize(vn[0], vs)
    ek[4, 1] = _brute_quantize(kn[2], ks)
    ev[4, 1] = _brute_quantize(vn[2], vs)
    assert (k2 == ek).all() and (v2 == ev).all()


def test_append_fp8_brute_force():
    check_append(oracle.append_kv_fp8)


# ------------------------------------------------------------- attention ---
def _fp8_case(seed, S, Hq, Hkv, D, BS, lens):
    rng = np.random.default_rng(seed)
    mb = max(1, max(-(-L // BS) for L in lens))
    nb = sum(-(-L // BS) for L in lens) + 2
    perm = rng.permutation(nb)
    table = -np.ones((S, mb), dtype=np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    codes = np.array(FINITE, dtype=np.uint8)
    kp = rng.choice(codes, (nb, BS, Hkv, D))
    vp = rng.choice(codes, (nb, BS, Hkv, D))
    return q, kp, vp, table, np.array(lens, dtype=np.int32)


def check_attention_closed_forms(attn):
    rng = np.random.default_rng(3)
    q, kp, vp, table, lens = _fp8_case(5, 2, 4, 2, 8, 4, [7, 1])
    ks = np.array([0.01, 0.02], dtype=np.float32)
    vs = np.array([0.5, 0.25], dtype=np.float32)
    # constant V code: every output row is that code's value times v_scale
    vc = np.full_like(vp, 0x3C)                              # 1.5
    out = attn(q, kp, vc, ks, vs, table, lens, np.float32(0.3))
    for h in range(4):
        assert np.allclose(out[:, h], 1.5 * float(vs[h // 2]), rtol=1e-12, atol=0)
    # one token: the output is that token's dequantized V row
    i = 1
    blk = table[i, 0]
    for h in range(4):
        exp = oracle.e4m3_decode(vp[blk, 0, h // 2]) * float(vs[h // 2])
        assert np.allclose(out_row(attn, q, kp, vp, ks, vs, table, lens)[i, h], exp,
                           rtol=1e-12, atol=1e-300)
    # equal K codes in a sequence: uniform weights, the mean of dequantized V
    kc = np.full_like(kp, int(rng.integers(0x30, 0x40)))
    o2 = attn(q, kc, vp, ks, vs, table, lens, np.float32(0.3))
    for h in range(4):
        rows = [oracle.e4m3_decode(vp[table[0, t // 4], t % 4, h // 2]) for t in range(7)]
        assert np.allclose(o2[0, h], np.mean(rows, axis=0) * float(vs[h // 2]), rtol=1e-12,
                           atol=1e-14)
    # k_scale multiplies the scores: doubling it doubles the effective softmax scale
    a = attn(q, kp, vp, ks * np.float32(2), vs, table, lens, np.float32(0.3))
    b = attn(q, kp, vp, ks, vs, table, lens, np.float32(0.6))
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def out_row(attn, q, kp, vp, ks, vs, table, lens):
    return attn(q, kp, vp, ks, vs, table, lens, np.float32(0.3))


def test_attention_fp8_closed_forms():
    check_attention_closed_forms(oracle.decode_attention_fp8)


def test_attention_fp8_brute_force():
    """Per-token loops over the dequantized cache in plain Python floats."""
    q, kp, vp, table, lens = _fp8_case(9, 2, 4, 2, 8, 4, [6, 9])
    ks = np.array([0.01, 0.02], dtype=np.float32)
    vs = np.array([0.5, 0.25], dtype=np.float32)
    sc = float(np.float32(0.35))
    out = oracle.decode_attention_fp8(q, kp, vp, ks, vs, table, lens, np.float32(0.35))
    for i in range(2):
        for h in range(4):
            kv = h // 2
            s = []
            for t in range(int(lens[i])):
                b, r = table[i, t // 4], t % 4
                s.append(sc * sum(float(q[i, h, d]) * float(oracle.e4m3_decode(kp[b, r, kv, d]))
                                  * float(ks[kv]) for d in range(8)))
            m = max(s)
            w = [np.exp(x - m) for x in s]
            z = sum(w)
            for d in range(8):
                acc = sum(w[t] * float(oracle.e4m3_decode(vp[table[i, t // 4], t % 4, kv, d]))
                          * float(vs[kv]) for t in range(int(lens[i])))
                assert abs(out[i, h, d] - acc / z) <= 1e-12 * max(1.0, abs(acc / z))


# ---------------------------------------------------------------- mutants ---
def _encode_truncating(x):
    a = np.asarray(x, dtype=np.float64).reshape(-1)
    out = np.empty(a.shape, dtype=np.uint8)
    for i, v in enumerate(a.tolist()):
        mag = min(abs(v), 448.0)
        code = int(np.searchsorted(f8._MAGS, mag, side="right")) - 1
        out[i] = code | (0x80 if v < 0 else 0)
    return out.reshape(np.asarray(x).shape)


def _encode_no_saturation(x):
    a = np.asarray(x, dtype=np.float64)
    out = oracle.e4m3_encode(a)
    return np.where(np.abs(a) > 448.0, np.uint8(0x7F), out).astype(np.uint8)


def _append_multiplying(kp, vp, kn, vn, slots, ks, vs):
    BS = kp.shape[1]
    k, v = kp.copy(), vp.copy()
    kq = oracle.e4m3_encode(kn.astype(np.float32) * ks.reshape(1, -1, 1))
    vq = oracle.e4m3_encode(vn.astype(np.float32) * vs.reshape(1, -1, 1))
    for i, s in enumerate(slots):
        if s >= 0:
            k[s // BS, s % BS], v[s // BS, s % BS] = kq[i], vq[i]
    return k, v


def _attn_scales_swapped(q, kp, vp, ks, vs, table, lens, scale):
    return oracle.decode_attention_fp8(q, kp, vp, vs, ks, table, lens, scale)


def _raises(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_mutant_truncating_encode_is_caught():
    assert _raises(lambda: check_ties_to_even(_encode_truncating, oracle.e4m3_decode))


def test_mutant_missing_saturation_is_caught():
    assert _raises(lambda: check_saturation(_encode_no_saturation))


def test_mutant_multiplying_append_is_caught():
    assert _raises(lambda: check_append(_append_multiplying))


def test_mutant_swapped_scales_is_caught():
    assert _raises(lambda: check_attention_closed_forms(_attn_scales_swapped))
