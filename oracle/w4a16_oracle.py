"""Plain CPU oracle for weight-only INT4 round-to-nearest quantization (W4A16).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers, tables or
pre/post-processing) and imports nothing from it.

What it computes, and where that is defined:

* "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
  the separation useful": weights are post-training quantized at load by
  round-to-nearest; the W4A16 preset stores attention and MLP projections as
  INT4 with group size 128 while activations stay BF16 (or FP16).
* The method specification that completes that description: symmetric codes
  in [-8, 7]; one fp16 scale per group of 128 consecutive K values, equal to
  the fp32 absmax of the group divided by 7; round-half-to-even; an all-zero
  group gets scale 1.
* "Piper Kernels", opening paragraphs: portable references compute in FP32
  rather than reproducing extra FP16/BF16 rounding; section "NVFP4
  construction": bias is applied in FP32 before the final output conversion,
  and projection tests compare against the independent reference on identical
  packed operands; section "ConvRot INT8": an MLP's SwiGLU of a raw
  [up | gate] tensor (``swiglu``, ``gemm_swiglu``).

Readings taken where the text leaves a step open (each one is listed with its
reason in the design notes of the repository):

1. Codes are computed from the *stored* fp16 scale, so that dequantize then
   requantize is idempotent.
2. ``x / s`` is an IEEE fp32 division, rounded to nearest even, and the
   quotient is then rounded to an integer with ties to even.
3. The zero rule is tested after the fp16 conversion: a scale that is zero in
   fp16 (all-zero group, or an absmax so small that absmax/7 underflows) is
   replaced by 1.0.
4. fp16 subnormal scales are kept (no flush to zero).
5. Packed layout: within a row, byte j holds code 2j in its low nibble and
   code 2j+1 in its high nibble, two's complement (``pack_codes`` gives the
   plain row-major ``[N, K/2]`` array).  The library stores those bytes in
   tiles of 128 rows x 128 K values (8 KiB, row-major inside the tile), tile
   (tn, g) at byte offset (tn * K/128 + g) * 8192, rows past N zero
   (``to_tile_layout`` / ``from_tile_layout``): a pure permutation of the
   row-major bytes.  ``scales[K/128, N]`` fp16, group-major.
6. Groups are contiguous runs of 128 along K, starting at k = 0, per row n.
7. Dequantized weight = float(code) * float(scale), exact in fp32.
8. GEMM: ``Y = A @ dequant(W)^T (+ bias)`` accumulated in FP32, bias added in
   FP32; the oracle returns the FP32 result (the library rounds it once to
   the activation type).
9. Activations, bias and output are BF16, or FP16 for the FP16-activation
   GEMM (the same page allows BF16 or FP16 activations); either widens to
   fp32 exactly.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
that do not come from this module: hand-worked examples, exact rational
arithmetic, brute force over all 16 codes and exact dot products.
"""

from __future__ import annotations

import numpy as np

GROUP = 128
QMIN = -8
QMAX = 7


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32.  Exact: bf16 is the top
    half of an IEEE binary32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen IEEE binary16 bit patterns (uint16) to float32 (exact)."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def act_bits_to_f32(bits: np.ndarray, act: str = "bf16") -> np.ndarray:
    """Activation bit patterns of type ``act`` ("bf16" or "f16") to float32."""
    if act == "bf16":
        return bf16_bits_to_f32(bits)
    if act == "f16":
        return f16_bits_to_f32(bits)
    raise ValueError(f"unknown activation type {act!r}")


def quantize_f32(x: np.ndarray, group: int = GROUP):
    """RTN-quantize a float32 weight ``x[N, K]``.

    Returns ``(packed uint8 [N, K/2], scale_bits uint16 [K/group, N])`` where
    ``scale_bits`` are IEEE binary16 bit patterns.  Steps, per row n and
    group g (k in [g*group, g*group + group)):

    1. amax = max |x|                  (fp32, exact)
    2. s32  = amax / 7                 (fp32 IEEE division, nearest-even)
    3. s    = fp16(s32)                (nearest-even, subnormals kept)
    4. s    = 1 if s == 0              (zero rule)
    5. q    = clamp(rint(x / s), -8, 7) with x / s an fp32 IEEE division
    6. pack two's-complement nibbles, low nibble = even k
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [N, K]")
    n_rows, k_cols = x.shape
    if group != GROUP:
        raise ValueError("only group size 128 is defined")
    if k_cols % group != 0:
        raise ValueError("K must be a multiple of the group size")
    n_groups = k_cols // group

    xg = x.reshape(n_rows, n_groups, group)
    amax = np.max(np.abs(xg), axis=2)                       # step 1
    s32 = amax / np.float32(7.0)                            # step 2
    s16 = s32.astype(np.float16)                            # step 3
    s16 = np.where(s16 == np.float16(0.0), np.float16(1.0), s16)  # step 4
    s_f32 = s16.astype(np.float32)                          # exact widening

    ratio = xg / s_f32[:, :, None]                          # step 5: fp32 divide
    q = np.clip(np.rint(ratio), QMIN, QMAX).astype(np.int8)
    codes = q.reshape(n_rows, k_cols)

    packed = pack_codes(codes)                              # step 6
    scale_bits = np.ascontiguousarray(s16.T).view(np.uint16)  # [G, N]
    return packed, scale_bits


def quantize(w_bits: np.ndarray, group: int = GROUP):
    """RTN-quantize a bf16 weight given as uint16 bit patterns ``[N, K]``."""
    return quantize_f32(bf16_bits_to_f32(w_bits), group)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Pack int codes ``[N, K]`` (values in [-8, 7]) into bytes ``[N, K/2]``:
    low nibble = even k, high nibble = odd k, two's complement."""
    c = np.asarray(codes).astype(np.int16)
    lo = (c[:, 0::2] & 0xF).astype(np.uint8)
    hi = (c[:, 1::2] & 0xF).astype(np.uint8)
    return (lo | (hi << np.uint8(4))).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_codes`: bytes ``[N, K/2]`` -> int8 codes ``[N, K]``."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    lo = (p & np.uint8(0xF)).astype(np.int16)
    hi = (p >> np.uint8(4)).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    n_rows, half = p.shape
    codes = np.empty((n_rows, 2 * half), dtype=np.int8)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    return codes


TILE_ROWS = 128      # rows of a storage tile
TILE_BYTES = TILE_ROWS * GROUP // 2


def tiled_bytes(n_rows: int, k_cols: int) -> int:
    """Bytes of the tiled storage of an [N, K] weight (rows padded to 128)."""
    return -(-n_rows // TILE_ROWS) * TILE_ROWS * k_cols // 2


def to_tile_layout(packed: np.ndarray) -> np.ndarray:
    """Row-major packed bytes [N, K/2] -> tiled storage (1-D uint8).
    Byte (n, j) goes to offset ((n // 128) * (K/128) + j // 64) * 8192 +
    (n % 128) * 64 + j % 64; padding rows are zero."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    n_rows, half = p.shape
    n_groups = half // (GROUP // 2)
    n_tiles = -(-n_rows // TILE_ROWS)
    padded = np.zeros((n_tiles * TILE_ROWS, half), dtype=np.uint8)
    padded[:n_rows] = p
    t = padded.reshape(n_tiles, TILE_ROWS, n_groups, GROUP // 2)   # [tn, r, g, byte]
    return np.ascontiguousarray(t.transpose(0, 2, 1, 3)).reshape(-1)


def from_tile_layout(tiled: np.ndarray, n_rows: int, k_cols: int) -> np.ndarray:
    """Inverse of :func:`to_tile_layout`: tiled storage -> [N, K/2] bytes."""
    b = np.ascontiguousarray(tiled, dtype=np.uint8).reshape(-1)
    n_tiles = -(-n_rows // TILE_ROWS)
    n_groups = k_cols // GROUP
    if b.size != n_tiles * TILE_ROWS * k_cols // 2:
        raise ValueError("tiled buffer has the wrong size")
    t = b.reshape(n_tiles, n_groups, TILE_ROWS, GROUP // 2).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(t.reshape(n_tiles * TILE_ROWS, k_cols // 2)[:n_rows])


def scales_f32(scale_bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns -> float32 (exact)."""
    return np.ascontiguousarray(scale_bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def dequantize(packed: np.ndarray, scale_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """``Wd[n, k] = float(q[n, k]) * float(scales[k // group, n])`` in fp32.
    The product of a 4-bit code and an 11-bit significand is exact."""
    codes = unpack_codes(packed).astype(np.float32)
    n_rows, k_cols = codes.shape
    s = scales_f32(scale_bits)                  # [G, N]
    if s.shape != (k_cols // group, n_rows):
        raise ValueError("scales must be [K/group, N]")
    s_nk = np.repeat(s.T, group, axis=1)        # [N, K]: scale of each element
    return codes * s_nk


def gemm(a_bits: np.ndarray, packed: np.ndarray, scale_bits: np.ndarray,
         bias_bits: np.ndarray | None = None, group: int = GROUP,
         rows: np.ndarray | None = None, act: str = "bf16") -> np.ndarray:
    """``Y[M, N] = A[M, K] @ dequant(W)[N, K]^T (+ bias[N])`` in FP32.

    ``a_bits`` and ``bias_bits`` are bit patterns of the activation type
    ``act`` ("bf16" or "f16").  ``rows`` (optional) selects the rows of A to
    evaluate, for sampled checks of large cases.  Returns float32; the
    library's output is that value rounded once to the activation type.
    """
    a = act_bits_to_f32(a_bits, act)
    if rows is not None:
        a = a[np.asarray(rows)]
    wd = dequantize(packed, scale_bits, group)
    if a.shape[1] != wd.shape[1]:
        raise ValueError("A and W disagree on K")
    y = np.matmul(a, wd.T, dtype=np.float32)
    if bias_bits is not None:
        y = y + act_bits_to_f32(bias_bits, act)[None, :]
    return y.astype(np.float32)


def swiglu(y: np.ndarray) -> np.ndarray:
    """SwiGLU of a pre-activation ``y[M, N]`` whose columns interleave up
    (even columns) and gate (odd columns): ``h[m, f] = silu(y[m, 2f + 1]) *
    y[m, 2f]`` with ``silu(g) = g / (1 + e^-g)``, in float64.

    "Piper Kernels", section "ConvRot INT8": the MLP's SwiGLU takes a raw
    [up | gate] tensor.  Interleaving the two halves column by column (up f,
    then gate f) is the reading that keeps each pair in one output tile, so
    the GEMM that produces them can apply SwiGLU before its one rounding.
    """
    y = np.asarray(y, dtype=np.float64)
    if y.shape[1] % 2 != 0:
        raise ValueError("N must be even (interleaved up and gate columns)")
    up, gate = y[:, 0::2], y[:, 1::2]
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


def gemm_swiglu(a_bits: np.ndarray, packed: np.ndarray, scale_bits: np.ndarray,
                bias_bits: np.ndarray | None = None, group: int = GROUP,
                rows: np.ndarray | None = None) -> np.ndarray:
    """``swiglu(gemm(...))``: the FP32 W4A16 GEMM with bf16 activations and
    bias, then SwiGLU of its interleaved up/gate columns (float64).  The
    library's output is that value rounded once to bf16."""
    return swiglu(gemm(a_bits, packed, scale_bits, bias_bits, group, rows))
