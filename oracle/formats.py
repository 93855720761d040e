"""Decoding of the element formats in a KV row.

FP8 e4m3 (OCP 8-bit floating point, E4M3 variant): sign, 4-bit exponent with
bias 7, 3-bit mantissa; exponent field 0 is subnormal (m * 2^-9); the codes
0x7F and 0xFF are NaN; there are no infinities. bf16: the upper 16 bits of an
IEEE binary32. The 656-byte row follows the ``fp8_ds_mla`` size in the
footnotes of "vLLM Part 2: PCP/DCP and P/D deployment with HiSparse"
(512 FP8 latent + 4 fp32 scales + 64 bf16 rope).
"""
import numpy as np

LATENT = 512
ROPE = 64
GROUP = 128


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = b >> 7
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def dequant_rows(rows: np.ndarray) -> np.ndarray:
    """[n, 656] uint8 -> [n, 576] float64: latent * group scale, then rope."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    lat = e4m3_to_f64(rows[:, :LATENT]).reshape(n, LATENT // GROUP, GROUP)
    scale = np.ascontiguousarray(rows[:, LATENT:LATENT + 16]).view("<f4").astype(np.float64)
    lat = (lat * scale[:, :, None]).reshape(n, LATENT)
    rope = bf16_to_f64(np.ascontiguousarray(rows[:, LATENT + 16:]).view("<u2"))
    return np.concatenate([lat, rope], axis=1)
