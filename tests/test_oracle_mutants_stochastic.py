"""Plants plausible mistakes in copies of the stochastic-rounding oracle (on
the CPU) and checks that at least one pin of test_oracle_stochastic fails for
each: a wrong Philox constant or round count, swapped key words, the wrong
output word, a transposed element offset, <= instead of <, a truncating
rounding, ratios taken against the unrounded fp32 scale.  (Rounding an
out-of-range value stochastically and then clamping is not a mistake: both
neighbours clamp to the same code as the deterministic result.)"""

import types

import numpy as np
import pytest

from oracle import stochastic as sr
import test_oracle_stochastic as T


def _philox(rounds=10, m0=sr.PHILOX_M0, swap_out=False):
    def f(ctr, key):
        c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint32) for c in ctr)
        k0 = np.asarray(key[0], dtype=np.uint32)
        k1 = np.asarray(key[1], dtype=np.uint32)
        with np.errstate(over="ignore"):
            for r in range(rounds):
                if r > 0:
                    k0 = (k0 + np.uint32(sr.PHILOX_W0)).astype(np.uint32)
                    k1 = (k1 + np.uint32(sr.PHILOX_W1)).astype(np.uint32)
                hi0, lo0 = sr._mulhilo(m0, c0)
                hi1, lo1 = sr._mulhilo(sr.PHILOX_M1, c2)
                c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        return (c1, c0, c2, c3) if swap_out else (c0, c1, c2, c3)
    return f


def _ns(philox=None, key_swap=False, word_shift=False, transposed=False, le=False,
        truncate=False, scale_fp32=False):
    ph = philox or sr.philox4x32_10

    def uniform_at(seed, offsets):
        e = np.asarray(offsets, dtype=np.uint64)
        c = e >> np.uint64(2)
        ctr = ((c & sr._MASK32).astype(np.uint32), (c >> np.uint64(32)).astype(np.uint32),
               np.zeros(e.shape, np.uint32), np.zeros(e.shape, np.uint32))
        k0, k1 = sr.seed_key(seed)
        words = np.stack(ph(ctr, (k1, k0) if key_swap else (k0, k1)))
        widx = ((e + np.uint64(1)) if word_shift else e) & np.uint64(3)
        w = np.take_along_axis(words, widx.astype(np.int64)[None], axis=0)[0]
        return ((w >> np.uint32(8)).astype(np.float32) * np.float32(2.0 ** -24)).astype(np.float32)

    def uniform_block(seed, k_cols, rows, cols):
        r = np.arange(rows.start, rows.stop, dtype=np.uint64)
        c = np.arange(cols.start, cols.stop, dtype=np.uint64)
        if transposed:
            return uniform_at(seed, r[:, None] + c[None, :] * np.uint64(1 << 20))
        return uniform_at(seed, r[:, None] * np.uint64(k_cols) + c[None, :])

    def stochastic_code(ratio, u):
        r = np.asarray(ratio, dtype=np.float32)
        u = np.asarray(u, dtype=np.float32)
        lo = np.trunc(r) if truncate else np.floor(r)
        frac = r - lo
        up = (u <= frac) if le else (u < frac)
        q = lo + up.astype(np.float32)
        det = np.clip(np.rint(r), -8, 7)
        interior = (r >= -8) & (r <= 7)
        return np.where(interior, q, det).astype(np.int8)

    def quantize_sr_f32(x, seed, group=128):
        x = np.ascontiguousarray(x, dtype=np.float32)
        n, k = x.shape
        xg = x.reshape(n, k // group, group)
        s32 = np.max(np.abs(xg), axis=2) / np.float32(7.0)
        s16 = s32.astype(np.float16)
        s16 = np.where(s16 == 0, np.float16(1.0), s16)
        sdiv = np.where(s32 == 0, np.float32(1.0), s32) if scale_fp32 else s16.astype(np.float32)
        ratio = (xg / sdiv[:, :, None]).reshape(n, k)
        codes = stochastic_code(ratio, uniform_block(seed, k, slice(0, n), slice(0, k)))
        return sr.pack_codes(codes), np.ascontiguousarray(s16.T).view(np.uint16)

    return types.SimpleNamespace(philox4x32_10=ph, uniform_at=uniform_at,
                                 uniform_block=uniform_block, stochastic_code=stochastic_code,
                                 quantize_sr_f32=quantize_sr_f32)


def _run_all(ns):
    for pin in T.ALL_PINS:
        pin(ns)


def test_unmutated_copy_passes():
    _run_all(_ns())


MUTANTS = {
    "rounds_7": dict(philox=_philox(rounds=7)),
    "multiplier": dict(philox=_philox(m0=0xD2511F55)),
    "output_order": dict(philox=_philox(swap_out=True)),
    "key_swap": dict(key_swap=True),
    "word_shift": dict(word_shift=True),
    "transposed_offset": dict(transposed=True),
    "le_instead_of_lt": dict(le=True),
    "scale_fp32": dict(scale_fp32=True),
    "truncate": dict(truncate=True),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_stochastic_mutant_is_caught(name):
    with pytest.raises(AssertionError):
        _run_all(_ns(**MUTANTS[name]))
