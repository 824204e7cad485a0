"""Seeded synthetic workloads for sink + low-rank recurrent-state decode.

This module is the one place that both the CPU oracle (through the tests) and
the GPU path take their inputs from. It holds no arithmetic of the method
itself: only a counter-based random number generator, the distributions of
the synthetic workloads, and their shapes.

Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11), written from its published definition.
The GPU library carries a device twin of the same generator and the same
counter layout (``include/seed_synth.h``); raw 32-bit outputs agree bit for
bit, and floats within a few ulp (the transcendental functions differ).

Counter layout, shared with the device twin:

    key     = (seed, (phase << 16) | field)
    counter = (block, time, entity, 0)

``block`` indexes groups of four values within one vector, ``time`` is the
prefill token or the decode step (0 for constants), ``entity`` is the
flattened head, the sink direction or the request, depending on the field.

Normals use the Box-Muller transform on pairs of uniforms: block ``b`` gives
values ``4b .. 4b+3`` from its four 32-bit words ``x0..x3`` as
``r(x0)cos(2 pi u(x1)), r(x0)sin(2 pi u(x1)), r(x2)cos(2 pi u(x3)),
r(x2)sin(2 pi u(x3))`` with ``r(x) = sqrt(-2 ln u(x))`` and
``u(x) = ((x >> 9) + 0.5) * 2**-23``, which lies strictly inside (0, 1) and
is exact in fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import numpy as np

# Philox4x32 multipliers and Weyl key increments (Salmon et al., SC'11, Table 2).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

# Phases of the counter layout.
PHASE_CONST = 0
PHASE_PREFILL = 1
PHASE_DECODE = 2

# Fields of the counter layout.  For Mamba-2 the read-out vector C uses the
# Q field, the input vector B the K field and the head input x the V field.
FIELD_Q = 1
FIELD_K = 2
FIELD_V = 3
FIELD_ALPHA = 4
FIELD_BETA = 5
FIELD_DT = 6
FIELD_VBAR = 16
FIELD_SINK_SCALE = 17
FIELD_A = 18
FIELD_RANK = 19
FIELD_CTX = 20


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on uint32 arrays (broadcast together).

    Each round multiplies words 0 and 2 by the two Philox constants, keeps
    the high and low halves of the 64-bit products, and mixes the high halves
    with the other two words and the round key; the key is advanced by the
    Weyl increments between rounds.  Returns the four output words.
    """
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(
        *(np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3, k0, k1)))
    c0, c1, c2, c3 = c0.copy(), c1.copy(), c2.copy(), c3.copy()
    k0, k1 = k0.copy(), k1.copy()
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        p0 = c0 * m0
        p1 = c2 * m1
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def field_key(phase: int, field: int) -> int:
    return ((phase & 0xFFFF) << 16) | (field & 0xFFFF)


def raw_words(seed: int, phase: int, field: int, time, entity, n_blocks: int) -> np.ndarray:
    """Raw generator words for blocks ``0..n_blocks-1``.

    ``time`` and ``entity`` broadcast against each other; the result has
    shape ``broadcast(time, entity).shape + (4 * n_blocks,)`` (uint32).
    """
    time = np.asarray(time, dtype=np.uint64)
    entity = np.asarray(entity, dtype=np.uint64)
    shape = np.broadcast_shapes(time.shape, entity.shape)
    blk = np.arange(n_blocks, dtype=np.uint64)
    t = np.broadcast_to(time, shape)[..., None]
    e = np.broadcast_to(entity, shape)[..., None]
    words = philox4x32_10(blk, t, e, 0, seed, field_key(phase, field))
    out = np.stack(words, axis=-1)  # [..., n_blocks, 4]
    return out.reshape(shape + (4 * n_blocks,))


def uniform_from_word(x: np.ndarray) -> np.ndarray:
    """Map 32-bit words to floats in (0, 1): ((x >> 9) + 1/2) * 2**-23 (exact in fp32)."""
    return (((x >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23)


def uniforms(seed, phase, field, time, entity, n) -> np.ndarray:
    """``n`` uniforms in (0, 1) per (time, entity); float64 values exact in fp32."""
    nb = (n + 3) // 4
    return uniform_from_word(raw_words(seed, phase, field, time, entity, nb))[..., :n]


def normals(seed, phase, field, time, entity, n) -> np.ndarray:
    """``n`` standard normals per (time, entity), rounded to fp32 (returned as float64)."""
    nb = (n + 3) // 4
    u = uniform_from_word(raw_words(seed, phase, field, time, entity, nb))
    u = u.reshape(u.shape[:-1] + (nb, 4))
    r01 = np.sqrt(-2.0 * np.log(u[..., 0]))
    r23 = np.sqrt(-2.0 * np.log(u[..., 2]))
    th01 = 2.0 * np.pi * u[..., 1]
    th23 = 2.0 * np.pi * u[..., 3]
    z = np.stack([r01 * np.cos(th01), r01 * np.sin(th01),
                  r23 * np.cos(th23), r23 * np.sin(th23)], axis=-1)
    z = z.reshape(z.shape[:-2] + (4 * nb,))[..., :n]
    return z.astype(np.float32).astype(np.float64)


def _f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _unit(z: np.ndarray) -> np.ndarray:
    return _f32(z / np.sqrt(np.sum(z * z, axis=-1, keepdims=True)))


def softplus(x):
    return np.log1p(np.exp(x))


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and input distributions of one synthetic decode workload.

    Heads are flattened as ``h = (request * n_layers + layer) * n_head + head``.
    Sink directions (and the per-direction sink scale and Mamba-2 ``A``) are
    per (layer, head) and shared by all requests: ``dir = h mod
    (n_layers * n_head)``.
    """
    name: str
    variant: str                 # 'gdn' | 'kda' | 'mamba2'
    n_req: int
    n_layers: int
    n_head: int
    d_k: int
    d_v: int
    T: int
    steps: int
    seed: int
    factor_dtype: str            # 'f32' | 'bf16' | 'f16'
    rank: int = 0                # uniform rank, or 0 when rank_choices is used
    rank_choices: Tuple[int, ...] = ()
    prefill_len: int = 0         # fixed prompt length, or 0 when prefill_range is used
    prefill_range: Tuple[int, int] = (0, 0)
    # value input v = s * vbar + noise_std * N(0, 1) (x for Mamba-2)
    sink_scale: Tuple[float, float] = (3.0, 3.0)   # U[lo, hi] per direction (lo == hi: constant)
    noise_std: float = 1.0
    alpha_range: Tuple[float, float] = (0.85, 0.999)
    beta_range: Tuple[float, float] = (0.05, 0.95)
    # Mamba-2: A = -U[a_lo, a_hi] per direction; dt = softplus(N(dt_mu, dt_var)); B, C ~ N(0, 1/N)
    a_range: Tuple[float, float] = (1.0, 16.0)
    dt_mu: float = -2.0
    dt_var: float = 0.5

    @property
    def n_heads(self) -> int:
        return self.n_req * self.n_layers * self.n_head

    @property
    def n_dir(self) -> int:
        return self.n_layers * self.n_head

    @property
    def growth(self) -> int:
        """Factor columns appended per decode step (two for the per-channel gate)."""
        return 2 if self.variant == 'kda' else 1

    @property
    def r_max(self) -> int:
        return max(self.rank_choices) if self.rank_choices else self.rank

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


GDN_TINY = Workload(
    name='gdn_tiny_b1_h4_r8', variant='gdn', n_req=1, n_layers=1, n_head=4, d_k=128, d_v=128,
    T=8, steps=64, seed=0, factor_dtype='f32', rank=8, prefill_len=256,
    sink_scale=(3.0, 3.0), noise_std=0.5, alpha_range=(0.9, 0.999), beta_range=(0.1, 0.9))

GDN_BATCHED = Workload(
    name='gdn_batched_b64_h32_r32', variant='gdn', n_req=64, n_layers=1, n_head=32, d_k=128,
    d_v=128, T=16, steps=256, seed=1, factor_dtype='bf16', rank=32, prefill_len=1024,
    sink_scale=(1.0, 4.0), noise_std=1.0, alpha_range=(0.85, 0.999), beta_range=(0.05, 0.95))

KDA_BATCHED = Workload(
    name='kda_batched_b128_h32_r32', variant='kda', n_req=128, n_layers=1, n_head=32, d_k=128,
    d_v=128, T=16, steps=512, seed=2, factor_dtype='bf16', rank=32, prefill_len=1024,
    sink_scale=(1.0, 4.0), noise_std=1.0, alpha_range=(0.8, 0.999), beta_range=(0.05, 0.95))

MAMBA2_BATCHED = Workload(
    name='mamba2_batched_b256_h128_r16', variant='mamba2', n_req=256, n_layers=1, n_head=128,
    d_k=128, d_v=64, T=16, steps=512, seed=3, factor_dtype='bf16', rank=16, prefill_len=2048,
    sink_scale=(2.0, 2.0), noise_std=1.0)

GDN_SERVING = Workload(
    name='gdn_serving_b512_l36_h32_ragged', variant='gdn', n_req=512, n_layers=36, n_head=32,
    d_k=128, d_v=128, T=16, steps=128, seed=4, factor_dtype='bf16', rank_choices=(16, 32, 48),
    prefill_range=(512, 8192), sink_scale=(1.0, 4.0), noise_std=1.0,
    alpha_range=(0.85, 0.999), beta_range=(0.05, 0.95))

WORKLOADS = {w.name: w for w in (GDN_TINY, GDN_BATCHED, KDA_BATCHED, MAMBA2_BATCHED, GDN_SERVING)}


# ----------------------------------------------------------------------------
# Per-direction, per-head and per-request constants
# ----------------------------------------------------------------------------

def sink_directions(w: Workload, dirs=None) -> np.ndarray:
    """Unit sink directions ``vbar`` (``xbar`` for Mamba-2), [n_dir, d_v]."""
    dirs = np.arange(w.n_dir) if dirs is None else np.asarray(dirs)
    return _unit(normals(w.seed, PHASE_CONST, FIELD_VBAR, 0, dirs, w.d_v))


def sink_scales(w: Workload, dirs=None) -> np.ndarray:
    dirs = np.arange(w.n_dir) if dirs is None else np.asarray(dirs)
    lo, hi = w.sink_scale
    u = uniforms(w.seed, PHASE_CONST, FIELD_SINK_SCALE, 0, dirs, 1)[..., 0]
    return _f32(lo + (hi - lo) * u)


def mamba2_A(w: Workload, dirs=None) -> np.ndarray:
    """Mamba-2 ``A = -U[a_lo, a_hi]`` per direction."""
    dirs = np.arange(w.n_dir) if dirs is None else np.asarray(dirs)
    lo, hi = w.a_range
    u = uniforms(w.seed, PHASE_CONST, FIELD_A, 0, dirs, 1)[..., 0]
    return _f32(-(lo + (hi - lo) * u))


def head_ranks(w: Workload, heads=None) -> np.ndarray:
    heads = np.arange(w.n_heads) if heads is None else np.asarray(heads)
    if not w.rank_choices:
        return np.full(np.shape(heads), w.rank, dtype=np.int32)
    x = raw_words(w.seed, PHASE_CONST, FIELD_RANK, 0, heads, 1)[..., 0]
    idx = (x.astype(np.uint64) * np.uint64(len(w.rank_choices))) >> np.uint64(32)
    return np.asarray(w.rank_choices, dtype=np.int32)[idx.astype(np.int64)]


def prompt_lengths(w: Workload, requests=None) -> np.ndarray:
    requests = np.arange(w.n_req) if requests is None else np.asarray(requests)
    if w.prefill_len:
        return np.full(np.shape(requests), w.prefill_len, dtype=np.int32)
    lo, hi = w.prefill_range
    x = raw_words(w.seed, PHASE_CONST, FIELD_CTX, 0, requests, 1)[..., 0]
    span = np.uint64(hi - lo + 1)
    return (lo + ((x.astype(np.uint64) * span) >> np.uint64(32))).astype(np.int32)


def head_dir(w: Workload, heads) -> np.ndarray:
    return np.asarray(heads) % w.n_dir


def head_request(w: Workload, heads) -> np.ndarray:
    return np.asarray(heads) // w.n_dir


# ----------------------------------------------------------------------------
# Per-token inputs
# ----------------------------------------------------------------------------

def token_inputs(w: Workload, phase: int, t, heads) -> dict:
    """Inputs of one token (prefill) or one decode step for the given heads.

    ``t`` and ``heads`` broadcast; every array gets that shape plus the
    vector length.  Values are fp32-representable, returned as float64.

    GDN / KDA: ``q, k`` (unit, [d_k]), ``v`` ([d_v]), ``alpha`` (scalar for
    GDN, [d_k] for KDA), ``beta`` (scalar).
    Mamba-2: ``C`` ([N]), ``B`` ([N]), ``x`` ([P]), ``dt`` (scalar).
    """
    heads = np.asarray(heads)
    t = np.asarray(t)
    dirs = head_dir(w, heads)
    vbar = sink_directions(w, dirs)
    if w.variant == 'mamba2':
        sd = 1.0 / math.sqrt(w.d_k)
        C = _f32(normals(w.seed, phase, FIELD_Q, t, heads, w.d_k) * sd)
        B = _f32(normals(w.seed, phase, FIELD_K, t, heads, w.d_k) * sd)
        xs = sink_scales(w, dirs)
        x = _f32(xs[..., None] * vbar + w.noise_std * normals(w.seed, phase, FIELD_V, t, heads, w.d_v))
        z = normals(w.seed, phase, FIELD_DT, t, heads, 1)[..., 0]
        dt = _f32(softplus(w.dt_mu + math.sqrt(w.dt_var) * z))
        return dict(C=C, B=B, x=x, dt=dt)
    q = _unit(normals(w.seed, phase, FIELD_Q, t, heads, w.d_k))
    k = _unit(normals(w.seed, phase, FIELD_K, t, heads, w.d_k))
    s = sink_scales(w, dirs)
    v = _f32(s[..., None] * vbar + w.noise_std * normals(w.seed, phase, FIELD_V, t, heads, w.d_v))
    alo, ahi = w.alpha_range
    blo, bhi = w.beta_range
    if w.variant == 'kda':
        alpha = _f32(alo + (ahi - alo) * uniforms(w.seed, phase, FIELD_ALPHA, t, heads, w.d_k))
    else:
        alpha = _f32(alo + (ahi - alo) * uniforms(w.seed, phase, FIELD_ALPHA, t, heads, 1)[..., 0])
    beta = _f32(blo + (bhi - blo) * uniforms(w.seed, phase, FIELD_BETA, t, heads, 1)[..., 0])
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta)


def decode_inputs(w: Workload, step: int, heads=None) -> dict:
    heads = np.arange(w.n_heads) if heads is None else np.asarray(heads)
    return token_inputs(w, PHASE_DECODE, step, heads)


def prefill_inputs(w: Workload, head: int, length: Optional[int] = None) -> dict:
    """All prompt-token inputs of one head, each array [L, ...]."""
    if length is None:
        length = int(prompt_lengths(w, [head // w.n_dir])[0])
    return token_inputs(w, PHASE_PREFILL, np.arange(length), np.full(length, head))


# ----------------------------------------------------------------------------
# Random factored states (for per-call parity tests)
# ----------------------------------------------------------------------------

def random_factored_state(seed: int, n_heads: int, d_k: int, d_v: int, m: Sequence[int],
                          cap: int, variant: str) -> dict:
    """Random sink + factor contents for testing single calls.

    Returns ``a`` [H, d_k], ``U`` [H, cap, d_k] and ``W`` [H, cap, d_v]
    (columns past ``m[h]`` are zero), ``scale`` [H, cap] in (0.3, 1] for the
    scalar-gate variants or ``D`` [H, d_k] in (0.3, 1] for the per-channel
    gate, and unit ``vbar`` [H, d_v].  All values fp32-representable.
    """
    m = np.asarray(m)
    heads = np.arange(n_heads)
    a = _f32(normals(seed, PHASE_CONST, 40, 0, heads, d_k))
    U = _f32(normals(seed, PHASE_CONST, 41, np.arange(cap)[None, :], heads[:, None], d_k) * 0.5)
    W = _f32(normals(seed, PHASE_CONST, 42, np.arange(cap)[None, :], heads[:, None], d_v) * 0.5)
    col = np.arange(cap)[None, :]
    U = U * (col < m[:, None])[..., None]
    W = W * (col < m[:, None])[..., None]
    vbar = _unit(normals(seed, PHASE_CONST, 43, 0, heads, d_v))
    out = dict(a=a, U=U, W=W, vbar=vbar)
    if variant == 'kda':
        out['D'] = _f32(0.3 + 0.7 * uniforms(seed, PHASE_CONST, 44, 0, heads, d_k))
    else:
        sc = _f32(0.3 + 0.7 * uniforms(seed, PHASE_CONST, 44, 0, heads, cap))
        out['scale'] = sc * (col < m[:, None])
    return out
