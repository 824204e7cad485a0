"""Algorithmic HBM bytes and FLOPs of the library's calls (for roofline figures).

Bytes are what the method must move per head and call, counted from the data
layout (``include/seed.h``): factor columns read once, appended columns,
sink coefficient, scales, per-step inputs and the output.  The per-direction
sink table is shared by all requests and stays in L2, so it is not counted
(the appendix accounting table of "Shallow Encoding Emits Deep Memories",
thelatestinai.com list view, also leaves the mean direction out).
"""
from __future__ import annotations

F32 = 4


def factor_bytes(factor_dtype: str) -> int:
    return 2 if factor_dtype in ('bf16', 'f16') else 4


def decode_bytes(variant: str, d_k: int, d_v: int, m: int, factor_dtype: str) -> int:
    """HBM bytes of one fused decode step of one head holding m columns."""
    s = factor_bytes(factor_dtype)
    cols = m * (d_k + d_v) * s                       # U and W read once
    a = 2 * d_k * F32                                # sink coefficient read + write
    if variant == 'gdn':
        ins = (2 * d_k + d_v + 2) * F32                # q, k, v, alpha, beta
        new = (d_k + d_v) * s                          # one appended column each
        sc = (m + (m + 1)) * F32                       # column scales read + write
    elif variant == 'kda':
        ins = (3 * d_k + d_v + 1) * F32                # q, k, v, alpha[d_k], beta
        new = 2 * (d_k + d_v) * s
        sc = 2 * d_k * F32                             # row scale D read + write
    else:
        ins = (2 * d_k + d_v + 1) * F32                # C, B, x, dt
        new = (d_k + d_v) * s
        sc = (m + (m + 1)) * F32
    out = d_v * F32
    return cols + a + ins + new + sc + out


def dense_decode_bytes(variant: str, d_k: int, d_v: int) -> int:
    """HBM bytes of one dense-state step of one head (state read + write, inputs, output)."""
    state = 2 * d_k * d_v * F32
    if variant == 'gdn':
        ins = (2 * d_k + d_v + 2) * F32
    elif variant == 'kda':
        ins = (3 * d_k + d_v + 1) * F32
    else:
        ins = (2 * d_k + d_v + 1) * F32
    return state + ins + d_v * F32


def recompress_bytes(variant: str, d_k: int, d_v: int, m: int, r: int, factor_dtype: str) -> int:
    s = factor_bytes(factor_dtype)
    sc = 2 * d_k * F32 if variant == 'kda' else (m + r) * F32
    return m * (d_k + d_v) * s + r * (d_k + d_v) * s + sc


def recompress_flops(d_k: int, d_v: int, m: int, r: int, sweeps: float) -> float:
    """FLOPs of one QR + core SVD recompression of one head with m columns.

    Householder QR of a p x m panel: 2 p m^2 - 2 m^3 / 3 (both factors);
    forming Q explicitly: the same again; core K = R_a R_b^T: 2 m^3 / 3;
    pivoted QR of the m x m core: 4 m^3 / 3; one Jacobi sweep: m (m - 1) / 2
    pairs, each three dot products of length m (6 m) and one rotation of a
    column pair (6 m), counted for every pair of every sweep; the kept
    directions through the core, K y_k: 2 m^2 r; rebuild of the r kept
    columns: 2 (d_k + d_v) m r.  This is the method's count; the three-phase
    kernels reach the same factors without forming Q and with scaled Jacobi
    rotations, so they execute fewer FLOPs than it.
    """
    qr = sum(2 * p * m * m - 2 * m ** 3 / 3 for p in (d_k, d_v))
    formq = qr
    core = 2 * m ** 3 / 3
    qrcp = 4 * m ** 3 / 3
    jac = sweeps * (m * (m - 1) / 2) * 12 * m
    kept = 2 * m * m * r
    rebuild = 2 * (d_k + d_v) * m * r
    return qr + formq + core + qrcp + jac + kept + rebuild
