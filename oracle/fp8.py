"""fp8 (E4M3) KV cache: the byte format, the quantizing append and attention
over a quantized cache.

Test infrastructure only (see the package docstring).

The pages name KV quantization as the way to shrink per-sequence KV and fit
more sequences ("Phase 7 · Document 04 — PagedAttention", §11 Engineering
Decision Framework: `--kv-cache-dtype fp8 (KV quant)`; §12 Hands-On Lab,
step 3). They fix no format. Readings taken here:

* Format: the OCP 8-bit floating point E4M3 encoding. Bit 7 is the sign,
  bits 6..3 the exponent (bias 7), bits 2..0 the mantissa. Exponent field 0
  encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities;
  the largest finite magnitude is 1.75 * 2^8 = 448.
* Scales: one fp32 scale per KV head for K and one for V. A cached value is
  code_value * scale.
* Quantizing (the append): the fp16 input widened to fp32 is divided by the
  head's scale in fp32 (IEEE, round to nearest even), and that fp32 quotient is
  rounded to the nearest E4M3 value, ties to the even code, magnitudes above
  448 saturating to 448 (NaN stays NaN).
* Attention over a quantized cache is the attention of the dequantized K and V
  (the plain definition in `attention.py`), computed in fp64.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_attention

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte(s) -> value(s) in fp64, from the bit fields."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = sign * (m / 8.0) * 2.0 ** -6
    out = np.where(e == 0, sub, normal)
    out = np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, out)
    return out


# the 127 finite non-negative magnitudes, code 0x00 .. 0x7E, increasing
_MAGS = e4m3_decode(np.arange(0x7F))


def e4m3_encode(x) -> np.ndarray:
    """Value(s) (taken exactly as given, normally fp32) -> E4M3 code(s):
    nearest value, ties to the even code, magnitudes past 448 -> 448, NaN ->
    0x7F, the sign kept (also for zero)."""
    a = np.asarray(x, dtype=np.float64)
    flat = a.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for i, v in enumerate(flat.tolist()):
        if v != v:
            out[i] = NAN_CODE
            continue
        neg = np.signbit(v)
        mag = abs(v)
        if mag >= E4M3_MAX:
            code = 0x7E
        else:
            hi = int(np.searchsorted(_MAGS, mag, side="left"))  # first magnitude >= mag
            if _MAGS[hi] == mag:
                code = hi
            else:
                lo = hi - 1
                dlo = mag - _MAGS[lo]
                dhi = _MAGS[hi] - mag
                if dlo < dhi:
                    code = lo
                elif dhi < dlo:
                    code = hi
                else:
                    code = lo if lo % 2 == 0 else hi
        out[i] = code | (0x80 if neg else 0)
    return out.reshape(a.shape)


def quantize_rows(x16: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """fp16 rows [..., Hkv, D] -> E4M3 codes with one fp32 scale per head:
    code(fp32(x) / scale[h]), the division in fp32."""
    x32 = np.asarray(x16, dtype=np.float16).astype(np.float32)
    s32 = np.asarray(scale, dtype=np.float32).reshape((1,) * (x32.ndim - 2) + (-1, 1))
    return e4m3_encode(np.divide(x32, s32, dtype=np.float32))


def append_kv_fp8(k_pool8: np.ndarray, v_pool8: np.ndarray, k_new: np.ndarray,
                  v_new: np.ndarray, slot_mapping, k_scale, v_scale) -> tuple:
    """Copies of the E4M3 pools [NB][BS][Hkv][D] with the quantized row i of
    k_new/v_new ([T][Hkv][D] fp16) at slot slot_mapping[i] (block slot // BS,
    row slot % BS); a negative slot writes nothing."""
    BS = k_pool8.shape[1]
    k = k_pool8.copy()
    v = v_pool8.copy()
    kq = quantize_rows(k_new, k_scale)
    vq = quantize_rows(v_new, v_scale)
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        k[slot // BS, slot % BS] = kq[i]
        v[slot // BS, slot % BS] = vq[i]
    return k, v


def dequantize_pool(pool8: np.ndarray, scale) -> np.ndarray:
    """E4M3 pool [NB][BS][Hkv][D] -> fp64 values, scale[h] applied per KV head."""
    s = np.asarray(scale, dtype=np.float32).astype(np.float64)
    return e4m3_decode(pool8) * s.reshape(1, 1, -1, 1)


class _DequantizedPool:
    """An E4M3 pool seen as its fp64 values; rows are decoded when indexed, so
    a sampled attention does not decode the whole pool."""

    def __init__(self, pool8: np.ndarray, scale):
        self.pool8 = pool8
        self.shape = pool8.shape
        self.scale = np.asarray(scale, dtype=np.float32).astype(np.float64).reshape(-1, 1)

    def __getitem__(self, idx):
        return e4m3_decode(self.pool8[idx]) * self.scale


def decode_attention_fp8(q, k_pool8, v_pool8, k_scale, v_scale, block_table, seq_lens, scale,
                         seqs=None, heads=None) -> np.ndarray:
    """Decode attention over E4M3 pools: the attention of the dequantized cache."""
    return decode_attention(q, _DequantizedPool(k_pool8, k_scale),
                            _DequantizedPool(v_pool8, v_scale), block_table, seq_lens, scale,
                            seqs=seqs, heads=heads)
