"""Plain CPU oracle for the seeded stochastic-rounding quantize mode.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library and imports nothing from it.

What it computes, and where that is defined:

* "Piper Kernels", section "Stochastic quantization": instead of the nearest
  code, one of the two adjacent codes is chosen with probability proportional
  to the distance between them, so the expected value is the unrounded one.
  Where a value is not interior to the representable range the deterministic
  result is used; values outside the range and exact hits on a code are never
  perturbed.  Draws come from a seeded generator (not a process-global one),
  indexed by the logical element offset, so the launch geometry cannot change
  which values are sampled and a caller replays a result by passing the same
  seed.
* Same page, section "ConvRot INT8" (the ``add_`` / ``addmm_`` weight
  updates): the seeded stochastic selection leaves the deterministic scales
  unchanged.
* The generator is Philox4x32-10, the counter-based generator published by
  Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3"
  (SC 2011): ten rounds of the Philox S-box on a 4 x 32-bit counter with a
  2 x 32-bit key; multipliers 0xD2511F53 and 0xCD9E8D57; Weyl key increments
  0x9E3779B9 and 0xBB67AE85 between rounds.

Readings taken where the text leaves a step open (listed with their reasons in
the design notes of the repository):

SR1. Scales are exactly the round-to-nearest scales: fp16(absmax / 7) with the
     zero rule (``w4a16_oracle.quantize_f32``).
SR2. The ratio r = x / s is the same IEEE fp32 division as in the
     round-to-nearest mode.  If r < -8 or r > 7 (not interior to the code
     range) the code is the deterministic one, clamp(rint(r), -8, 7).
     Otherwise lo = floor(r) and frac = r - lo (exact in fp32), and the code is
     lo + 1 when u < frac, else lo; an exact hit (frac = 0) is never perturbed.
SR3. u for element (n, k) of the logical [N, K] weight: e = n * K + k;
     Philox4x32-10 with key (seed mod 2^32, seed div 2^32) on the counter
     (c mod 2^32, c div 2^32, 0, 0) with c = e div 4; word (e mod 4) of the
     result, w; u = (w >> 8) * 2^-24, a float32 in [0, 1) held exactly.

Every function here is pinned by ``tests/test_oracle_stochastic.py``: the
published known-answer vectors of Philox4x32-10, the unbiasedness of the
rounding, brute force over explicit draws and the invariants the page states.
"""

from __future__ import annotations

import numpy as np

from .w4a16_oracle import GROUP, QMAX, QMIN, bf16_bits_to_f32, pack_codes

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10
_MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(m: int, x: np.ndarray):
    """32 x 32 -> 64-bit product of the constant m and the uint32 values x:
    (high word, low word)."""
    p = np.uint64(m) * x.astype(np.uint64)
    return (p >> np.uint64(32)).astype(np.uint32), (p & _MASK32).astype(np.uint32)


def philox4x32_10(ctr, key):
    """Philox4x32-10 applied to counters ``ctr`` (four uint32 arrays of one
    shape) under ``key`` (two uint32 values or arrays).  Returns four uint32
    arrays.

    One round maps (c0, c1, c2, c3) under (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is advanced by the Weyl constants before every round but the
    first."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint32) for c in ctr)
    k0 = np.asarray(key[0], dtype=np.uint32)
    k1 = np.asarray(key[1], dtype=np.uint32)
    with np.errstate(over="ignore"):
        for r in range(PHILOX_ROUNDS):
            if r > 0:
                k0 = (k0 + np.uint32(PHILOX_W0)).astype(np.uint32)
                k1 = (k1 + np.uint32(PHILOX_W1)).astype(np.uint32)
            hi0, lo0 = _mulhilo(PHILOX_M0, c0)
            hi1, lo1 = _mulhilo(PHILOX_M1, c2)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def seed_key(seed: int):
    """Key words of a 64-bit seed (reading SR3)."""
    seed = int(seed)
    if not 0 <= seed < (1 << 64):
        raise ValueError("seed must be an unsigned 64-bit integer")
    return np.uint32(seed & 0xFFFFFFFF), np.uint32(seed >> 32)


def uniform_at(seed: int, offsets: np.ndarray) -> np.ndarray:
    """u in [0, 1) (float32) for the logical element offsets ``offsets``
    (reading SR3): the draw depends on the seed and the offset only."""
    e = np.asarray(offsets, dtype=np.uint64)
    c = e >> np.uint64(2)
    ctr = ((c & _MASK32).astype(np.uint32), (c >> np.uint64(32)).astype(np.uint32),
           np.zeros(e.shape, np.uint32), np.zeros(e.shape, np.uint32))
    words = np.stack(philox4x32_10(ctr, seed_key(seed)))      # [4, ...]
    w = np.take_along_axis(words, (e & np.uint64(3)).astype(np.int64)[None], axis=0)[0]
    return ((w >> np.uint32(8)).astype(np.float32) * np.float32(2.0 ** -24)).astype(np.float32)


def uniform_block(seed: int, k_cols: int, rows: slice, cols: slice) -> np.ndarray:
    """u for the block ``[rows, cols]`` of a logical [N, k_cols] weight."""
    r = np.arange(rows.start, rows.stop, dtype=np.uint64)
    c = np.arange(cols.start, cols.stop, dtype=np.uint64)
    return uniform_at(seed, r[:, None] * np.uint64(k_cols) + c[None, :])


def stochastic_code(ratio: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Codes from fp32 ratios r = x / s and draws u (reading SR2)."""
    r = np.asarray(ratio, dtype=np.float32)
    u = np.asarray(u, dtype=np.float32)
    lo = np.floor(r)
    frac = r - lo                                  # exact: |r| < 2^23
    up = u < frac
    sr = lo + up.astype(np.float32)
    det = np.clip(np.rint(r), QMIN, QMAX)
    interior = (r >= np.float32(QMIN)) & (r <= np.float32(QMAX))
    return np.where(interior, sr, det).astype(np.int8)


def quantize_sr_f32(x: np.ndarray, seed: int, group: int = GROUP, row0: int = 0):
    """Stochastic-rounding quantize of a float32 weight ``x[N, K]``
    (``row0``: ``x`` holds rows row0 .. row0 + N - 1 of a larger logical
    weight; the draws follow the logical offsets).

    Returns ``(packed uint8 [N, K/2], scale_bits uint16 [K/group, N])``.
    Steps, per row n and group g:

    1. amax, s32 = amax / 7, s = fp16(s32), s = 1 if s == 0 (the RTN scale)
    2. r = x / s (fp32 IEEE division)
    3. u = the Philox draw of element (n, k)
    4. q = stochastic_code(r, u)
    5. pack two's-complement nibbles, low nibble = even k
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [N, K]")
    if group != GROUP:
        raise ValueError("only group size 128 is defined")
    n_rows, k_cols = x.shape
    if k_cols % group != 0:
        raise ValueError("K must be a multiple of the group size")
    n_groups = k_cols // group
    xg = x.reshape(n_rows, n_groups, group)
    amax = np.max(np.abs(xg), axis=2)                            # step 1
    s16 = (amax / np.float32(7.0)).astype(np.float16)
    s16 = np.where(s16 == np.float16(0.0), np.float16(1.0), s16)
    ratio = (xg / s16.astype(np.float32)[:, :, None]).reshape(n_rows, k_cols)   # step 2
    u = uniform_block(seed, k_cols, slice(row0, row0 + n_rows), slice(0, k_cols))  # step 3
    codes = stochastic_code(ratio, u)                                           # step 4
    return pack_codes(codes), np.ascontiguousarray(s16.T).view(np.uint16)       # step 5


def quantize_sr(w_bits: np.ndarray, seed: int, group: int = GROUP, row0: int = 0):
    """Stochastic-rounding quantize of a bf16 weight (uint16 bit patterns)."""
    return quantize_sr_f32(bf16_bits_to_f32(w_bits), seed, group, row0)
