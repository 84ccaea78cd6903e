"""Shared helpers of the GPU parity tests: oracle calls on the CPU and the
GEMM tolerance |y - y_ref| <= 1e-2 |y_ref| + 1e-2 rms(y_ref)."""

import numpy as np
import torch

import oracle
from weight_only_int4_rtn_gb300 import synthetic

REL_TOL = 1e-2
RMS_TOL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return synthetic.bits(t.detach().cpu())


def oracle_quantize(W: torch.Tensor):
    return oracle.quantize(bits(W))


def check_quantize_exact(W: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor):
    p_rm, s_ref = oracle_quantize(W)
    p_ref = oracle.to_tile_layout(p_rm)
    p = packed.cpu().numpy().reshape(-1)
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    assert p.shape == p_ref.shape and s.shape == s_ref.shape
    bad_s = np.argwhere(s != s_ref)
    assert bad_s.size == 0, f"{len(bad_s)} scale mismatches, first {bad_s[:4].tolist()}"
    bad_p = np.argwhere(p != p_ref)
    assert bad_p.size == 0, f"{len(bad_p)} packed-byte mismatches, first {bad_p[:4].tolist()}"


def check_gemm_close(y: torch.Tensor, y_ref: np.ndarray, rms: float | None = None, what=""):
    yg = y.float().cpu().numpy()
    assert yg.shape == y_ref.shape, (yg.shape, y_ref.shape)
    assert np.isfinite(yg).all(), f"{what}: non-finite output"
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref.astype(np.float64) ** 2)))
    err = np.abs(yg.astype(np.float64) - y_ref)
    lim = REL_TOL * np.abs(y_ref) + RMS_TOL * rms
    bad = np.argwhere(err > lim)
    assert bad.size == 0, (
        f"{what}: {len(bad)} of {err.size} outside tolerance; worst excess "
        f"{float(np.max(err - lim)):.4g} at {bad[:3].tolist()}")
    return float(np.max(err / (np.abs(y_ref) + rms + 1e-30)))


def guarded(shape, dtype, device, fill_bits: int, slack: int = 256):
    """A tensor of `shape` that sits inside a larger buffer whose slack is
    filled with a sentinel; returns (view, checker)."""
    n = int(np.prod(shape))
    elem = torch.empty(0, dtype=dtype).element_size()
    raw = torch.empty(n + 2 * slack, dtype=dtype, device=device)
    if elem == 2:
        raw.view(torch.int16).fill_(np.int16(np.uint16(fill_bits).view(np.int16)))
    else:
        raw.view(torch.uint8).fill_(fill_bits & 0xFF)
    view = raw[slack:slack + n].view(shape)

    def untouched():
        head = raw[:slack].cpu()
        tail = raw[slack + n:].cpu()
        ref = raw.new_empty(slack).cpu()
        if elem == 2:
            ref.view(torch.int16).fill_(np.int16(np.uint16(fill_bits).view(np.int16)))
            return torch.equal(head.view(torch.int16), ref.view(torch.int16)) and \
                torch.equal(tail.view(torch.int16), ref.view(torch.int16))
        ref.view(torch.uint8).fill_(fill_bits & 0xFF)
        return torch.equal(head, ref) and torch.equal(tail, ref)

    return view, untouched
