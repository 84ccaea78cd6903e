"""Plain CPU oracle for the FP4 weight-only schemes (MXFP4 and NVFP4) with
BF16 activations.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library and imports nothing from it.

What it computes, and where that is defined:

* "Kernel dispatch and Humming quantization in PhyAI", section "Choose
  precision by layer and hardware": MXFP4 and NVFP4 are among the Humming
  weight schemes, with BF16 activations.
* "Piper Kernels", section "NVFP4 construction": NVFP4 weights are built
  from a floating-point weight with blocks of 16 values and a per-tensor
  scale; section "NVFP4 construction" and the opening paragraphs: scales
  are applied in FP32, references compute in FP32.
* The element format of both is FP4 E2M1 (sign, two exponent bits with bias
  1, one mantissa bit): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
* MXFP4 follows the OCP Microscaling (MX) formats specification v1.0: blocks
  of 32 values share an E8M0 scale 2^(E - 127), with
  E = floor(log2(amax)) - 2 + 127 (2 is the exponent of the largest E2M1
  value, 6 = 1.5 * 2^2); elements are V / 2^(E - 127) rounded to nearest
  even in E2M1 and saturated to +-6.

Readings taken where the text leaves a step open (listed with their reasons in
the design notes of the repository):

F4-1. E2M1 rounding: nearest representable value, ties to the even mantissa
      bit; magnitudes above 6 saturate to 6; the sign is kept (-0 -> +0).
F4-2. MXFP4 all-zero block: E = 127 (scale 1), codes 0.  E is clamped to
      [0, 254].
F4-3. NVFP4: tensor scale g = fl32(amax_tensor / 2688) (2688 = 6 * 448, the
      largest E2M1 times the largest E4M3), g = 1 when amax_tensor is 0;
      block scale: the one-level scale fl32(amax_b / 6) expressed in units of
      g, s_b = e4m3_rn_sat(fl32(fl32(amax_b / 6) / g)) (E4M3 with bias 7,
      three mantissa bits, subnormals, largest 448, round to nearest even,
      saturating); codes e2m1(fl32(x / fl32(s_b * g))), codes 0 when
      s_b * g is 0.  Dequantized weight = code * s_b * g.
F4-4. Storage: codes as nibbles exactly like the INT4 codes (byte j of row n
      holds k = 2j in its low nibble, 2j + 1 in its high nibble; sign in the
      nibble's top bit, then exponent, then mantissa), in the same 8 KiB
      tiles.  Scales as bytes ``[K/32, N]`` (MXFP4, E8M0) or ``[K/16, N]``
      (NVFP4, E4M3) plus the fp32 tensor scale.

Pinned by ``tests/test_oracle_fp4.py``: the E2M1 and E4M3 value sets from the
format definitions with brute-force nearest-even rounding, the MX exponent by
exact arithmetic, hand-worked blocks, dequantize exactness and the GEMM
against exact dot products.
"""

from __future__ import annotations

import numpy as np

from .w4a16_oracle import act_bits_to_f32, bf16_bits_to_f32

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)
E2M1_MAX = np.float32(6.0)
E4M3_MAX = 448.0
NV_TENSOR_DEN = np.float32(2688.0)   # 6 * 448
MX_BLOCK = 32
NV_BLOCK = 16


# ---------------------------------------------------------------- formats
def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of 4-bit E2M1 codes (uint8 0..15): sign bit 3, magnitude index
    bits 0..2 (exponent bits 2..1, mantissa bit 0)."""
    c = np.asarray(codes, np.uint8)
    mag = E2M1_MAG[c & 7]
    return np.where((c & 8) != 0, -mag, mag).astype(np.float32)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Reading F4-1: nearest E2M1 value, ties to the even mantissa bit,
    saturating at 6.  Implemented as thresholds between neighbouring
    magnitudes (each midpoint goes to the neighbour with mantissa 0)."""
    a = np.abs(np.asarray(x, np.float32))
    # midpoints between magnitudes i and i+1, and which side a tie takes
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    tie_up = np.array([False, True, False, True, False, True, False])   # upper neighbour has mantissa 0
    idx = np.zeros(a.shape, np.uint8)
    for i, (m, up) in enumerate(zip(mids, tie_up)):
        idx = np.where((a > m) | ((a == m) & up), np.uint8(i + 1), idx)
    neg = np.signbit(np.asarray(x, np.float32)) & (idx != 0)
    return (idx | (neg.astype(np.uint8) << 3)).astype(np.uint8)


def e4m3_values() -> np.ndarray:
    """All finite non-negative E4M3 values, by code 0..126 (bias 7, three
    mantissa bits; code 0x7F is NaN)."""
    out = []
    for c in range(127):
        e, m = c >> 3, c & 7
        out.append((m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(out, np.float64)


_E4M3 = e4m3_values()


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Non-negative float32 values to E4M3 codes: nearest value, ties to the
    even code (even mantissa), saturating at 448."""
    v = np.asarray(x, np.float64)
    codes = np.searchsorted(_E4M3, v)               # first value >= v
    codes = np.clip(codes, 0, 126)
    lo = np.clip(codes - 1, 0, 126)
    d_hi = np.abs(_E4M3[codes] - v)
    d_lo = np.abs(v - _E4M3[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    out = np.where(pick_lo, lo, codes)
    out = np.where(v >= E4M3_MAX, 126, out)
    return out.astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _E4M3[np.asarray(codes, np.int64)].astype(np.float32)


# ---------------------------------------------------------------- MXFP4
def mx_exponent(amax: np.ndarray) -> np.ndarray:
    """E8M0 exponent code of a block: floor(log2(amax)) - 2 + 127, clamped
    to [0, 254]; 127 for amax = 0 (reading F4-2).  floor(log2) is exact from
    the float's own exponent (frexp)."""
    a = np.asarray(amax, np.float64)
    m, e = np.frexp(a)                 # a = m * 2^e, m in [0.5, 1)
    fl = e - 1                         # floor(log2(a)) for a > 0
    code = np.clip(fl - 2 + 127, 0, 254)
    return np.where(a == 0, 127, code).astype(np.uint8)


def quantize_mxfp4_f32(x: np.ndarray):
    """MXFP4 quantize of a float32 weight ``x[N, K]`` (K a multiple of 128).
    Returns ``(packed uint8 [N, K/2], scale_codes uint8 [K/32, N])``."""
    x = np.ascontiguousarray(x, np.float32)
    n, k = x.shape
    if k % 128:
        raise ValueError("K must be a multiple of 128")
    xb = x.reshape(n, k // MX_BLOCK, MX_BLOCK)
    e = mx_exponent(np.max(np.abs(xb), axis=2))                         # [N, K/32]
    scale = np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(np.float32)
    codes = e2m1_encode(xb / scale[:, :, None]).reshape(n, k)            # exact division
    return pack_codes_fp4(codes), np.ascontiguousarray(e.T)


def dequantize_mxfp4(packed: np.ndarray, scale_codes: np.ndarray) -> np.ndarray:
    codes = unpack_codes_fp4(packed)
    n, k = codes.shape
    s = np.ldexp(np.float32(1.0), scale_codes.astype(np.int32).T - 127).astype(np.float32)  # [N, K/32]
    return (e2m1_decode(codes) * np.repeat(s, MX_BLOCK, axis=1)).astype(np.float32)


# ---------------------------------------------------------------- NVFP4
def nv_tensor_scale(x: np.ndarray) -> np.float32:
    amax = np.float32(np.max(np.abs(np.asarray(x, np.float32)))) if np.size(x) else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(amax / NV_TENSOR_DEN)


def quantize_nvfp4_f32(x: np.ndarray, tensor_scale: np.float32 | None = None):
    """NVFP4 quantize of a float32 weight ``x[N, K]`` (reading F4-3).
    Returns ``(packed uint8 [N, K/2], scale_codes uint8 [K/16, N], g fp32)``."""
    x = np.ascontiguousarray(x, np.float32)
    n, k = x.shape
    if k % 128:
        raise ValueError("K must be a multiple of 128")
    g = nv_tensor_scale(x) if tensor_scale is None else np.float32(tensor_scale)
    xb = x.reshape(n, k // NV_BLOCK, NV_BLOCK)
    amax = np.max(np.abs(xb), axis=2)                                    # [N, K/16]
    one_level = (amax / np.float32(E2M1_MAX)).astype(np.float32)
    sb_code = e4m3_encode((one_level / g).astype(np.float32))
    sb = e4m3_decode(sb_code)
    step = (sb * g).astype(np.float32)                                   # fl32(s_b * g)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(step[:, :, None] > 0, xb / step[:, :, None], np.float32(0.0)).astype(np.float32)
    codes = e2m1_encode(r).reshape(n, k)
    return pack_codes_fp4(codes), np.ascontiguousarray(sb_code.T), g


def dequantize_nvfp4(packed: np.ndarray, scale_codes: np.ndarray, g: np.float32) -> np.ndarray:
    """code * s_b * g in float64 rounded once to float32 (the GEMM applies g
    in fp32 to the accumulated sum)."""
    codes = unpack_codes_fp4(packed)
    sb = e4m3_decode(scale_codes).astype(np.float64).T                   # [N, K/16]
    v = e2m1_decode(codes).astype(np.float64) * np.repeat(sb, NV_BLOCK, axis=1) * float(g)
    return v.astype(np.float32)


# ---------------------------------------------------------------- packing
def pack_codes_fp4(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [N, K] (uint8 0..15) -> bytes [N, K/2], low nibble = even k."""
    c = np.asarray(codes, np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes_fp4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


# ---------------------------------------------------------------- GEMM
def gemm_fp4(a_bits: np.ndarray, wd: np.ndarray, bias_bits: np.ndarray | None = None,
             rows=None) -> np.ndarray:
    """``Y = A @ Wd^T (+ bias)`` in FP32 with bf16 activations, Wd the
    dequantized weight of either scheme."""
    a = act_bits_to_f32(a_bits, "bf16")
    if rows is not None:
        wd = wd[rows]
    y = a @ wd.T
    if bias_bits is not None:
        b = bf16_bits_to_f32(bias_bits)
        y = y + (b if rows is None else b[rows])[None, :]
    return y.astype(np.float32)
