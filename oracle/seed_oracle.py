"""Plain float64 oracle of the SEED decode-time state path (test infrastructure only).

Sources, cited by page title and section:

* [summary] "Shallow Encoding Emits Deep Memories", picx.dev markdown summary:
  Methodology > "Roofline Cost Model", "SEED Architecture" (decode paragraph:
  S = a vbar^T + U V^T), "Exact Update (Lemma 2)", "Open-Loop Error Bound
  (Corollary 4)"; Theoretical and Practical Implications > "Lemma 1 (sink
  decomposition)".
* [list view] "Shallow Encoding Emits Deep Memories", thelatestinai.com list
  view: Table 1 (decode column: read-out and update of each recurrent state,
  compression to rank R every W steps, compression at the end of prefill),
  Table 2 (state at R / mean / peak MB, resident request MB), the drift table
  (state bytes as a share of dense fp32) and the appendix accounting table
  (the mean direction is shared by all requests and not counted).

Notation follows the summary page: the value-side factor that the page calls
V is called W here, the decay g is the gate (alpha for the delta rules,
exp(dt*A) for Mamba-2), the key kappa is k (B for Mamba-2).

Readings where the pages leave a step open:

* the read-out uses the state after the step's update (o_t = S_t^T q_t);
* the per-channel gate follows diag(alpha)(I - beta k k^T) S + beta k v^T,
  which the factored form follows exactly by appending two columns per step;
* the gate of the scalar-gate variants is kept as a per-column scale c
  (U diag(c) W^T), and the per-channel gate as a row scale D (diag(D) U W^T),
  so that existing columns are never rewritten;
* compression keeps a = S vbar / |vbar|^2 exactly and truncates the content
  C = S - a vbar^T by its SVD; the singular values go with U (U = X_r Sigma_r,
  W = Y_r) and the scales reset to one;
* recompression runs after step t when t is a multiple of T; the step's
  output uses the state before it.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

__all__ = [
    'FactoredState', 'gdn_dense_step', 'kda_dense_step', 'mamba2_dense_step', 'dense_step',
    'dense_prefill', 'sink_split', 'compress_dense', 'materialize', 'readout',
    'gdn_factored_step', 'kda_factored_step', 'mamba2_factored_step', 'factored_step',
    'recompress', 'state_bytes', 'dense_state_bytes', 'open_loop_bound', 'rel_fro',
    'run_head', 'HeadTrajectory',
]


# ----------------------------------------------------------------------------
# Dense recurrences (the original model's state path)
# ----------------------------------------------------------------------------

def gdn_dense_step(S, q, k, v, alpha, beta):
    """Gated DeltaNet: S' = alpha (I - beta k k^T) S + beta k v^T, o = S'^T q.

    [summary] Introduction: each linear-attention head keeps one d_k x d_v
    recurrent state; the update is the gated delta rule of the Gated DeltaNet
    layers that Lemma 2 covers.  (I - beta k k^T) S is written S - beta k (k^T S).
    """
    S = np.asarray(S, np.float64)
    kS = k @ S
    S_new = alpha * (S - beta * np.outer(k, kS)) + beta * np.outer(k, v)
    return S_new, S_new.T @ q


def kda_dense_step(S, q, k, v, alpha, beta):
    """Kimi Delta Attention with a per-channel gate alpha in R^{d_k}:
    S' = diag(alpha) (I - beta k k^T) S + beta k v^T, o = S'^T q."""
    S = np.asarray(S, np.float64)
    kS = k @ S
    S_new = alpha[:, None] * (S - beta * np.outer(k, kS)) + beta * np.outer(k, v)
    return S_new, S_new.T @ q


def mamba2_dense_step(S, C, B, x, dt, A):
    """Mamba-2 (N x P state): S' = exp(dt A) S + dt B x^T, y = S'^T C."""
    S = np.asarray(S, np.float64)
    g = math.exp(dt * A)
    S_new = g * S + dt * np.outer(B, x)
    return S_new, S_new.T @ C


def dense_step(variant: str, S, tok: Dict[str, np.ndarray], A: Optional[float] = None):
    if variant == 'gdn':
        return gdn_dense_step(S, tok['q'], tok['k'], tok['v'], float(tok['alpha']), float(tok['beta']))
    if variant == 'kda':
        return kda_dense_step(S, tok['q'], tok['k'], tok['v'], np.asarray(tok['alpha']), float(tok['beta']))
    if variant == 'mamba2':
        return mamba2_dense_step(S, tok['C'], tok['B'], tok['x'], float(tok['dt']), float(A))
    raise ValueError(variant)


def _token(tokens: Dict[str, np.ndarray], t: int) -> Dict[str, np.ndarray]:
    return {name: arr[t] for name, arr in tokens.items()}


def dense_prefill(variant: str, tokens: Dict[str, np.ndarray], d_k: int, d_v: int,
                  A: Optional[float] = None, S0=None) -> np.ndarray:
    """Run the dense recurrence over the prompt tokens from S = 0 (or S0).

    [list view] Table 1: the states that leave the prefill are compressed at
    its end, so the prefill itself is the plain recurrence over the prompt.
    """
    S = np.zeros((d_k, d_v)) if S0 is None else np.array(S0, np.float64)
    L = len(next(iter(tokens.values())))
    for t in range(L):
        S, _ = dense_step(variant, S, _token(tokens, t), A)
    return S


# ----------------------------------------------------------------------------
# Sink + low-rank state
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class FactoredState:
    """S = a vbar^T + U_eff W^T ([summary] SEED Architecture, decode paragraph).

    ``U`` is the stored key-side factor [d_k, m] and ``W`` the value-side
    factor [d_v, m].  The effective key factor is ``U diag(scale)`` for the
    scalar-gate variants (``scale`` [m]) and ``diag(D) U`` for the per-channel
    gate (``D`` [d_k]).  ``vbar`` is the fixed sink direction [d_v].
    """
    a: np.ndarray
    U: np.ndarray
    W: np.ndarray
    vbar: np.ndarray
    scale: Optional[np.ndarray] = None
    D: Optional[np.ndarray] = None

    @property
    def m(self) -> int:
        return self.U.shape[1]

    def U_eff(self) -> np.ndarray:
        if self.D is not None:
            return self.D[:, None] * self.U
        return self.U * self.scale[None, :]

    def copy(self) -> "FactoredState":
        return FactoredState(*(None if x is None else np.array(x, np.float64) for x in
                               (self.a, self.U, self.W, self.vbar, self.scale, self.D)))


def materialize(st: FactoredState) -> np.ndarray:
    """S = a vbar^T + U_eff W^T."""
    return np.outer(st.a, st.vbar) + st.U_eff() @ st.W.T


def readout(st: FactoredState, q) -> np.ndarray:
    """o = S^T q = vbar (a^T q) + W (U_eff^T q), without forming S."""
    return st.vbar * (st.a @ q) + st.W @ (st.U_eff().T @ q)


def sink_split(S, vbar):
    """Lemma 1 split of a state along vbar: a = S vbar / |vbar|^2, C = S - a vbar^T.

    [summary] Lemma 1 (sink decomposition): splitting each value along the
    fixed direction vbar separates the sink coefficient a from the content C,
    and C vbar = 0.
    """
    S = np.asarray(S, np.float64)
    a = S @ vbar / (vbar @ vbar)
    return a, S - np.outer(a, vbar)


def _truncate_svd(M, r):
    """Best rank-r factors of M by its SVD: (X_r Sigma_r, Y_r, discarded energy)."""
    X, s, Yt = np.linalg.svd(M, full_matrices=False)
    r_eff = min(r, len(s))
    U = X[:, :r_eff] * s[:r_eff]
    W = Yt[:r_eff].T
    err = float(np.sqrt(np.sum(s[r_eff:] ** 2)))
    return U, W, err, s


def compress_dense(S, vbar, r: int, variant: str = 'gdn'):
    """Dense state -> sink + rank-r factors.

    [list view] Table 1: the states that leave the prefill are compressed to
    the sink plus rank-R factors.  a = S vbar / |vbar|^2 (Lemma 1), content
    C = S - a vbar^T truncated to rank r by its SVD.  Returns (state, error)
    with error = |C - U W^T|_F.
    """
    vbar = np.asarray(vbar, np.float64)
    a, C = sink_split(S, vbar)
    U, W, err, _ = _truncate_svd(C, r)
    st = FactoredState(a=a, U=U, W=W, vbar=vbar.copy())
    if variant == 'kda':
        st.D = np.ones(len(a))
    else:
        st.scale = np.ones(U.shape[1])
    return st, err


def _omega_eps(v, vbar):
    """omega = v^T vbar / |vbar|^2 and eps = v - omega vbar ([summary] Lemma 2)."""
    omega = (v @ vbar) / (vbar @ vbar)
    return omega, v - omega * vbar


def gdn_factored_step(st: FactoredState, q, k, v, alpha, beta):
    """One Gated DeltaNet step on the factors ([summary] Exact Update (Lemma 2)).

    With g = alpha and kappa = k:
        a+ = g a + beta (omega - g k^T a) k
        U+ = [g U, k]                       (g goes into the column scales)
        W+ = [W, beta (eps - g W U^T k)]    (U here is the effective U diag(c))
    Returns the new state and the read-out of the updated state at q.
    """
    g = float(alpha)
    omega, eps = _omega_eps(v, st.vbar)
    Ue = st.U_eff()
    a_new = g * st.a + beta * (omega - g * (k @ st.a)) * k
    w_new = beta * (eps - g * (st.W @ (Ue.T @ k)))
    new = FactoredState(a=a_new, U=np.column_stack([st.U, k]), W=np.column_stack([st.W, w_new]),
                        vbar=st.vbar, scale=np.append(g * st.scale, 1.0))
    return new, readout(new, q)


def kda_factored_step(st: FactoredState, q, k, v, alpha, beta):
    """One Kimi Delta Attention step on the factors, gate diag(alpha) after the erase.

    S' = diag(alpha) S - beta (alpha*k)(k^T S) + beta k v^T.  Split with
    Lemma 1 and keep the gate as the row scale D (U_eff = diag(D) U):
        a+ = alpha * (a - beta k (k^T a)) + beta omega k
        D+ = alpha * D
        U+ = [U, k / D, k / D+]             (so that diag(D+) U+ = [diag(alpha) U_eff, alpha*k, k])
        W+ = [W, -beta W (U_eff^T k), beta eps]
    Two columns per step; exact ([summary] Lemma 2 covers the per-channel gate).
    """
    alpha = np.asarray(alpha, np.float64)
    omega, eps = _omega_eps(v, st.vbar)
    x_k = st.U_eff().T @ k
    a_new = alpha * (st.a - beta * k * (k @ st.a)) + beta * omega * k
    D_new = alpha * st.D
    U_new = np.column_stack([st.U, k / st.D, k / D_new])
    W_new = np.column_stack([st.W, -beta * (st.W @ x_k), beta * eps])
    new = FactoredState(a=a_new, U=U_new, W=W_new, vbar=st.vbar, D=D_new)
    return new, readout(new, q)


def mamba2_factored_step(st: FactoredState, C, B, x, dt, A):
    """One Mamba-2 step on the factors: S' = g S + dt B x^T with g = exp(dt A).

    No erase term, so Lemma 2 reduces to
        a+ = g a + dt omega B,   U+ = [g U, dt B],   W+ = [W, eps]
    with omega = x^T xbar / |xbar|^2, eps = x - omega xbar; y = S'^T C.
    """
    g = math.exp(float(dt) * float(A))
    omega, eps = _omega_eps(x, st.vbar)
    a_new = g * st.a + dt * omega * B
    new = FactoredState(a=a_new, U=np.column_stack([st.U, dt * B]), W=np.column_stack([st.W, eps]),
                        vbar=st.vbar, scale=np.append(g * st.scale, 1.0))
    return new, readout(new, C)


def factored_step(variant: str, st: FactoredState, tok: Dict[str, np.ndarray], A: Optional[float] = None):
    if variant == 'gdn':
        return gdn_factored_step(st, tok['q'], tok['k'], tok['v'], float(tok['alpha']), float(tok['beta']))
    if variant == 'kda':
        return kda_factored_step(st, tok['q'], tok['k'], tok['v'], np.asarray(tok['alpha']), float(tok['beta']))
    if variant == 'mamba2':
        return mamba2_factored_step(st, tok['C'], tok['B'], tok['x'], float(tok['dt']), float(A))
    raise ValueError(variant)


def recompress(st: FactoredState, r: int):
    """Compress the factors back to rank r ([list view] Table 1, every W steps).

    A = U_eff, B = W; thin QR A = Q_a R_a, B = Q_b R_b; core K = R_a R_b^T;
    SVD K = X Sigma Y^T; keep the r largest: U = Q_a X_r Sigma_r, W = Q_b Y_r;
    scales (or D) reset to one; a is unchanged.  Returns (state, error) with
    error = sqrt(sum of the discarded sigma^2) = |U_eff W^T - U' W'^T|_F.
    """
    Qa, Ra = np.linalg.qr(st.U_eff())
    Qb, Rb = np.linalg.qr(st.W)
    K = Ra @ Rb.T
    X, s, Yt, = np.linalg.svd(K)
    r_eff = min(r, len(s))
    U = Qa @ (X[:, :r_eff] * s[:r_eff])
    W = Qb @ Yt[:r_eff].T
    err = float(np.sqrt(np.sum(s[r_eff:] ** 2)))
    new = FactoredState(a=st.a.copy(), U=U, W=W, vbar=st.vbar)
    if st.D is not None:
        new.D = np.ones_like(st.D)
    else:
        new.scale = np.ones(r_eff)
    return new, err


# ----------------------------------------------------------------------------
# Accounting and bounds
# ----------------------------------------------------------------------------

def state_bytes(d_k: int, d_v: int, m: int, bytes_per_elem: float) -> float:
    """Bytes of one head's shallow state with m factor columns.

    [list view] appendix accounting table: the shallow state is the sink's
    coefficient (d_k numbers) and the factors ((d_k + d_v) m numbers); the
    mean direction is shared by all requests and not counted.
    """
    return bytes_per_elem * ((d_k + d_v) * m + d_k)


def dense_state_bytes(d_k: int, d_v: int, bytes_per_elem: float) -> float:
    """Bytes of one dense d_k x d_v head state."""
    return bytes_per_elem * d_k * d_v


def open_loop_bound(eps_bar: float, g_bar: float, W: int) -> float:
    """Corollary 4 ([summary] Open-Loop Error Bound): |S~_t - S_t|_F <= eps_bar / (1 - g_bar^W)."""
    return eps_bar / (1.0 - g_bar ** W)


def rel_fro(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / np.linalg.norm(ref))


# ----------------------------------------------------------------------------
# One head through prefill, compression and the decode loop
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class HeadTrajectory:
    outputs: List[np.ndarray]            # o_t (y_t), t = 1..steps
    states: Dict[int, np.ndarray]        # reconstructed dense state after step t (before recompression)
    compress_errors: List[float]         # error of compress_dense, then of each recompression
    prefill_state: np.ndarray
    final: FactoredState


def run_head(variant: str, prefill_state: np.ndarray, vbar, r: int, T: int,
             step_tokens: Callable[[int], Dict[str, np.ndarray]], steps: int,
             A: Optional[float] = None, record_states: Sequence[int] = (),
             compress: bool = True) -> HeadTrajectory:
    """Decode one head from a dense prefill state.

    [list view] Table 1: compress at the end of the prefill, then every step
    read out and update the factors, and compress back to rank r every T
    steps (after step t when T divides t).  ``step_tokens(t)`` gives the
    inputs of decode step t (0-based).  With ``compress=False`` the factors
    grow without truncation after the initial compression.
    """
    st, e0 = compress_dense(prefill_state, vbar, r, variant)
    errs = [e0]
    outs: List[np.ndarray] = []
    states: Dict[int, np.ndarray] = {}
    rec = set(record_states)
    for t in range(1, steps + 1):
        st, o = factored_step(variant, st, step_tokens(t - 1), A)
        outs.append(o)
        if t in rec:
            states[t] = materialize(st)
        if compress and t % T == 0:
            st, e = recompress(st, r)
            errs.append(e)
    return HeadTrajectory(outputs=outs, states=states, compress_errors=errs,
                          prefill_state=np.array(prefill_state, np.float64), final=st)
