"""Plain CPU oracle for weight-only INT8 round-to-nearest quantization (W8A16).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library and imports nothing from it.

What it computes, and where that is defined:

* "Kernel dispatch and Humming quantization in PhyAI", section "Choose
  precision by layer and hardware": the Humming integration supports INT4,
  INT8, FP8, MXFP4 and NVFP4 weight schemes with BF16 activations; section
  "Humming makes the separation useful": round-to-nearest quantization at
  load, group size 128, activations stay BF16 (or FP16), and the packed
  layout runs only through the kernel that understands it.
* "Piper Kernels", opening paragraphs and section "NVFP4 construction":
  portable references compute in FP32; bias is applied in FP32 before the
  final output conversion.

Readings taken where the text leaves a step open (listed with their reasons in
the design notes of the repository):

W8-1. The INT8 scheme is the INT4 method with 8-bit codes: symmetric codes in
      [-128, 127]; one fp16 scale per group of 128 consecutive K values,
      s = fp16(fp32 absmax / 127), replaced by 1 when it is 0; codes
      q = clamp(rint_even(fl32(x / s)), -128, 127) from the stored scale.
W8-2. Storage: one two's-complement byte per code.  The library keeps the
      bytes in tiles of 128 rows x 128 K values (16 KiB, row-major inside:
      128 B per row), tile (tn, g) at byte offset (tn * K/128 + g) * 16384,
      rows past N (to the next multiple of 128) zero; ``to_tile_layout8`` is
      that permutation of the row-major ``[N, K]`` bytes.  Scales
      ``[K/128, N]`` fp16, group-major, as for INT4.
W8-3. Dequantized weight = float(q) * float(s), exact in fp32 (8-bit x 11-bit
      significands); GEMM ``Y = A @ dequant(W)^T (+ bias)`` accumulated in
      FP32 with the bias added in FP32.

Pinned by ``tests/test_oracle_w8a16.py``: hand-worked groups, brute force over
all 256 codes, exact rational scales, invariants and exact dot products.
"""

from __future__ import annotations

import numpy as np

from .w4a16_oracle import GROUP, act_bits_to_f32, bf16_bits_to_f32, scales_f32

Q8MIN = -128
Q8MAX = 127
TILE8_BYTES = 128 * 128


def quantize8_f32(x: np.ndarray, group: int = GROUP):
    """RTN-quantize a float32 weight ``x[N, K]`` to INT8 codes.

    Returns ``(codes uint8 [N, K] (two's complement), scale_bits uint16
    [K/group, N])``.  Steps, per row n and group g:

    1. amax = max |x|                  (fp32, exact)
    2. s32  = amax / 127               (fp32 IEEE division, nearest-even)
    3. s    = fp16(s32)                (nearest-even, subnormals kept)
    4. s    = 1 if s == 0              (zero rule)
    5. q    = clamp(rint(x / s), -128, 127), x / s an fp32 IEEE division
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [N, K]")
    if group != GROUP:
        raise ValueError("only group size 128 is defined")
    n_rows, k_cols = x.shape
    if k_cols % group != 0:
        raise ValueError("K must be a multiple of the group size")
    xg = x.reshape(n_rows, k_cols // group, group)
    amax = np.max(np.abs(xg), axis=2)                              # step 1
    s16 = (amax / np.float32(127.0)).astype(np.float16)            # steps 2, 3
    s16 = np.where(s16 == np.float16(0.0), np.float16(1.0), s16)   # step 4
    ratio = xg / s16.astype(np.float32)[:, :, None]                # step 5
    q = np.clip(np.rint(ratio), Q8MIN, Q8MAX).astype(np.int8).reshape(n_rows, k_cols)
    return q.view(np.uint8), np.ascontiguousarray(s16.T).view(np.uint16)


def quantize8(w_bits: np.ndarray, group: int = GROUP):
    """RTN INT8 quantize of a bf16 weight given as uint16 bit patterns."""
    return quantize8_f32(bf16_bits_to_f32(w_bits), group)


def tiled8_bytes(n_rows: int, k_cols: int) -> int:
    """Bytes of the tiled INT8 storage of an [N, K] weight (rows padded to 128)."""
    return ((n_rows + 127) // 128) * 128 * k_cols


def to_tile_layout8(codes: np.ndarray) -> np.ndarray:
    """Row-major code bytes [N, K] -> tiled storage (1-D uint8), reading W8-2."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    n_rows, k_cols = codes.shape
    n_tiles = (n_rows + 127) // 128
    padded = np.zeros((n_tiles * 128, k_cols), np.uint8)
    padded[:n_rows] = codes
    g = k_cols // 128
    t = padded.reshape(n_tiles, 128, g, 128).transpose(0, 2, 1, 3)   # [tn, g, row, k]
    return np.ascontiguousarray(t).reshape(-1)


def from_tile_layout8(tiled: np.ndarray, n_rows: int, k_cols: int) -> np.ndarray:
    """Inverse of :func:`to_tile_layout8`: tiled storage -> [N, K] bytes."""
    n_tiles = (n_rows + 127) // 128
    g = k_cols // 128
    t = np.asarray(tiled, np.uint8).reshape(n_tiles, g, 128, 128).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(t).reshape(n_tiles * 128, k_cols)[:n_rows]


def dequantize8(codes: np.ndarray, scale_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """``Wd[n, k] = float(q[n, k]) * float(scales[k // group, n])`` in fp32."""
    q = np.ascontiguousarray(codes, np.uint8).view(np.int8).astype(np.float32)
    s = scales_f32(scale_bits)                       # [G, N]
    return q * np.repeat(s.T, group, axis=1)


def gemm8(a_bits: np.ndarray, codes: np.ndarray, scale_bits: np.ndarray,
          bias_bits: np.ndarray | None = None, group: int = GROUP, rows=None,
          act: str = "bf16") -> np.ndarray:
    """``Y[M, N] = A[M, K] @ dequant8(W)[N, K]^T (+ bias[N])`` in FP32 (the
    library rounds it once to the activation type).  ``rows`` restricts the
    output to a subset of weight rows."""
    a = act_bits_to_f32(a_bits, act)
    if rows is not None:
        codes = np.asarray(codes)[rows]
        scale_bits = np.asarray(scale_bits)[:, rows]
    wd = dequantize8(codes, scale_bits, group)
    y = a @ wd.T
    if bias_bits is not None:
        b = act_bits_to_f32(bias_bits, act)
        y = y + (b if rows is None else b[rows])[None, :]
    return y.astype(np.float32)
