"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values
computed by hand, closed forms, answers known by construction, brute force
on tiny inputs, the pages' printed numbers, and the pages' error bound.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), 'golden')


# ----------------------------------------------------------------------------
# helpers owned by the tests (no oracle arithmetic)
# ----------------------------------------------------------------------------

def householder_orthogonal(n, rng, n_reflectors=None):
    """Orthogonal n x n matrix as a product of Householder reflectors I - 2 u u^T / u^T u."""
    Q = np.eye(n)
    for _ in range(n if n_reflectors is None else n_reflectors):
        u = rng.standard_normal(n)
        Q = Q - 2.0 * np.outer(Q @ u, u) / (u @ u)
    return Q


def unit(x):
    return x / np.linalg.norm(x)


# ----------------------------------------------------------------------------
# dense recurrences: values computed by hand
# ----------------------------------------------------------------------------

S2 = np.array([[1.0, 2.0], [3.0, 4.0]])


def test_gdn_dense_hand_example():
    # k = e0, v = (5, 6), alpha = beta = 1/2, q = e1:
    # S - beta k (k^T S) = [[0.5, 1], [3, 4]]; times alpha: [[0.25, 0.5], [1.5, 2]];
    # plus beta k v^T = [[2.5, 3], [0, 0]]  ->  [[2.75, 3.5], [1.5, 2]]; o = row 1.
    S_new, o = oracle.gdn_dense_step(S2, np.array([0.0, 1.0]), np.array([1.0, 0.0]),
                                     np.array([5.0, 6.0]), 0.5, 0.5)
    assert np.allclose(S_new, [[2.75, 3.5], [1.5, 2.0]], atol=0, rtol=1e-15)
    assert np.allclose(o, [1.5, 2.0], atol=0, rtol=1e-15)


def test_kda_dense_hand_example():
    # same as above with alpha = (1/2, 1/4) applied to the rows after the erase
    S_new, o = oracle.kda_dense_step(S2, np.array([0.0, 1.0]), np.array([1.0, 0.0]),
                                     np.array([5.0, 6.0]), np.array([0.5, 0.25]), 0.5)
    assert np.allclose(S_new, [[2.75, 3.5], [0.75, 1.0]], atol=0, rtol=1e-15)
    assert np.allclose(o, [0.75, 1.0], atol=0, rtol=1e-15)


def test_mamba2_dense_hand_example():
    # dt = 1/2, A = -2 ln 2 -> exp(dt A) = 1/2; B = (2, 0), x = (1, 1), C = (1, 1):
    # S' = S/2 + [[1, 1], [0, 0]] = [[1.5, 2], [1.5, 2]]; y = S'^T C = (3, 4)
    S_new, y = oracle.mamba2_dense_step(S2, np.array([1.0, 1.0]), np.array([2.0, 0.0]),
                                        np.array([1.0, 1.0]), 0.5, -2.0 * math.log(2.0))
    assert np.allclose(S_new, [[1.5, 2.0], [1.5, 2.0]], atol=1e-15)
    assert np.allclose(y, [3.0, 4.0], atol=1e-14)


def test_delta_rule_writes_value_at_key():
    # alpha = beta = 1, unit k: k^T S' = k^T (I - k k^T) S + v^T = v^T (the delta rule stores v at k)
    rng = np.random.default_rng(0)
    S = rng.standard_normal((16, 12))
    k = unit(rng.standard_normal(16))
    v = rng.standard_normal(12)
    S_new, _ = oracle.gdn_dense_step(S, k, k, v, 1.0, 1.0)
    assert np.allclose(k @ S_new, v, atol=1e-12)
    S_new, _ = oracle.kda_dense_step(S, k, k, v, np.ones(16), 1.0)
    assert np.allclose(k @ S_new, v, atol=1e-12)


def test_dense_special_cases():
    rng = np.random.default_rng(1)
    S = rng.standard_normal((8, 6))
    q, k = unit(rng.standard_normal(8)), unit(rng.standard_normal(8))
    v = rng.standard_normal(6)
    # beta = 0: pure decay
    S_new, _ = oracle.gdn_dense_step(S, q, k, v, 0.7, 0.0)
    assert np.allclose(S_new, 0.7 * S, atol=1e-15)
    # per-channel gate with equal channels is the scalar gate
    a1, o1 = oracle.gdn_dense_step(S, q, k, v, 0.8, 0.3)
    a2, o2 = oracle.kda_dense_step(S, q, k, v, np.full(8, 0.8), 0.3)
    assert np.allclose(a1, a2, atol=1e-14) and np.allclose(o1, o2, atol=1e-14)
    # Mamba-2 with A = 0 adds dt B x^T; dt -> 0 leaves S
    S_new, _ = oracle.mamba2_dense_step(S, q, k, v, 0.25, 0.0)
    assert np.allclose(S_new, S + 0.25 * np.outer(k, v), atol=1e-14)
    S_new, _ = oracle.mamba2_dense_step(S, q, k, v, 0.0, -3.0)
    assert np.allclose(S_new, S, atol=0)


def test_gdn_erase_removes_component_along_key():
    # beta = 1, v = 0: S' = alpha (I - k k^T) S kills k^T S exactly
    rng = np.random.default_rng(2)
    S = rng.standard_normal((10, 7))
    k = unit(rng.standard_normal(10))
    S_new, _ = oracle.gdn_dense_step(S, k, k, np.zeros(7), 0.9, 1.0)
    assert np.allclose(k @ S_new, 0, atol=1e-13)
    # and leaves components orthogonal to k scaled by alpha
    p = rng.standard_normal(10)
    p -= (p @ k) * k
    assert np.allclose(p @ S_new, 0.9 * (p @ S), atol=1e-13)


# ----------------------------------------------------------------------------
# factored update (Lemma 2): exact against the dense recurrence
# ----------------------------------------------------------------------------

def _small_workload(variant, d_k=16, d_v=12):
    base = {'gdn': synth.GDN_BATCHED, 'kda': synth.KDA_BATCHED, 'mamba2': synth.MAMBA2_BATCHED}[variant]
    return base.with_(n_req=1, n_head=3, d_k=d_k, d_v=d_v, rank=4, T=4, steps=40, prefill_len=24)


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_factored_equals_dense_without_compression(variant):
    w = _small_workload(variant)
    for h in range(w.n_heads):
        d = synth.head_dir(w, h)
        vbar = synth.sink_directions(w, [d])[0]
        A = float(synth.mamba2_A(w, [d])[0]) if variant == 'mamba2' else None
        S = oracle.dense_prefill(variant, synth.prefill_inputs(w, h), w.d_k, w.d_v, A)
        st, _ = oracle.compress_dense(S, vbar, w.rank, variant)
        S_dense = oracle.materialize(st)
        for t in range(w.steps):
            tok = {kk: vv[0] for kk, vv in synth.token_inputs(w, synth.PHASE_DECODE, t, [h]).items()}
            st, o = oracle.factored_step(variant, st, tok, A)
            S_dense, o_dense = oracle.dense_step(variant, S_dense, tok, A)
            assert oracle.rel_fro(oracle.materialize(st), S_dense) < 1e-12
            assert oracle.rel_fro(o, o_dense) < 1e-11
        assert st.m == w.rank + w.growth * w.steps


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_sink_split_invariants_lemma1(variant):
    # From a compressed state, W^T vbar = 0 and a = S vbar / |vbar|^2 after every step.
    w = _small_workload(variant)
    h = 1
    d = synth.head_dir(w, h)
    vbar = synth.sink_directions(w, [d])[0]
    A = float(synth.mamba2_A(w, [d])[0]) if variant == 'mamba2' else None
    S = oracle.dense_prefill(variant, synth.prefill_inputs(w, h), w.d_k, w.d_v, A)
    st, _ = oracle.compress_dense(S, vbar, w.rank, variant)
    for t in range(12):
        tok = {kk: vv[0] for kk, vv in synth.token_inputs(w, synth.PHASE_DECODE, t, [h]).items()}
        st, _ = oracle.factored_step(variant, st, tok, A)
        scale = np.linalg.norm(st.W)
        assert np.max(np.abs(st.W.T @ vbar)) < 1e-13 * max(scale, 1.0)
        a_split, _ = oracle.sink_split(oracle.materialize(st), vbar)
        assert np.allclose(a_split, st.a, atol=1e-12 * np.linalg.norm(st.a))


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_readout_is_state_transpose_times_query(variant):
    w = _small_workload(variant)
    rng = np.random.default_rng(3)
    vbar = unit(rng.standard_normal(w.d_v))
    S = rng.standard_normal((w.d_k, w.d_v))
    st, _ = oracle.compress_dense(S, vbar, 5, variant)
    tok = {kk: vv[0] for kk, vv in synth.token_inputs(w, synth.PHASE_DECODE, 0, [0]).items()}
    st, o = oracle.factored_step(variant, st, tok, -1.5 if variant == 'mamba2' else None)
    q = tok['C'] if variant == 'mamba2' else tok['q']
    assert np.allclose(o, oracle.materialize(st).T @ q, atol=1e-12)


def test_factored_delta_rule_property():
    rng = np.random.default_rng(4)
    vbar = unit(rng.standard_normal(12))
    S = rng.standard_normal((16, 12))
    st, _ = oracle.compress_dense(S, vbar, 16)          # exact (rank <= 12)
    k = unit(rng.standard_normal(16))
    v = rng.standard_normal(12)
    st, o = oracle.gdn_factored_step(st, k, k, v, 1.0, 1.0)
    assert np.allclose(o, v, atol=1e-12)                # read-out at the key returns the value


# ----------------------------------------------------------------------------
# compression: Eckart-Young by construction, closed form, brute force
# ----------------------------------------------------------------------------

def _constructed_state(d_k, d_v, sigma, rng):
    """S = a0 vbar^T + X diag(sigma) Y^T with Y^T vbar = 0, all known by construction."""
    n = len(sigma)
    Qx = householder_orthogonal(d_k, rng)
    Qv = householder_orthogonal(d_v, rng)
    vbar = Qv[:, 0]
    X = Qx[:, :n]
    Y = Qv[:, 1:n + 1]
    a0 = rng.standard_normal(d_k)
    S = np.outer(a0, vbar) + (X * sigma) @ Y.T
    return S, a0, vbar, X, Y


@pytest.mark.parametrize('r', [1, 3, 5])
def test_compress_dense_constructed(r):
    rng = np.random.default_rng(10 + r)
    sigma = np.array([9.0, 7.0, 4.0, 2.5, 1.5, 0.75, 0.25])
    S, a0, vbar, X, Y = _constructed_state(12, 10, sigma, rng)
    st, err = oracle.compress_dense(S, vbar, r)
    assert np.allclose(st.a, a0, atol=1e-12)
    expect = np.outer(a0, vbar) + (X[:, :r] * sigma[:r]) @ Y[:, :r].T
    assert oracle.rel_fro(oracle.materialize(st), expect) < 1e-12
    assert err == pytest.approx(math.sqrt(np.sum(sigma[r:] ** 2)), rel=1e-12)
    assert np.allclose(np.sort(np.linalg.norm(st.U, axis=0))[::-1], sigma[:r], rtol=1e-12)


def test_compress_dense_closed_form_2x3():
    # d_k = 2, d_v = 3: the content lies in the 2-dim complement of vbar; the rank-1
    # truncation error is the smaller singular value, from the 2x2 closed form
    # sigma^2 = (t -/+ sqrt(t^2 - 4 det)) / 2 of C C^T.
    S = np.array([[1.0, -2.0, 0.5], [3.0, 1.0, -1.0]])
    vbar = np.array([1.0, 1.0, 1.0]) / math.sqrt(3.0)
    st, err = oracle.compress_dense(S, vbar, 1)
    a = S.sum(axis=1) / math.sqrt(3.0)
    C = S - np.outer(a, vbar)
    g00, g01, g11 = C[0] @ C[0], C[0] @ C[1], C[1] @ C[1]
    t, det = g00 + g11, g00 * g11 - g01 * g01
    lam_min = (t - math.sqrt(t * t - 4 * det)) / 2
    assert np.allclose(st.a, a, atol=1e-14)
    assert err == pytest.approx(math.sqrt(lam_min), rel=1e-10)
    assert oracle.rel_fro(oracle.materialize(st), S) == pytest.approx(math.sqrt(lam_min) / np.linalg.norm(S), rel=1e-10)


def test_compress_full_rank_is_exact():
    rng = np.random.default_rng(5)
    S = rng.standard_normal((9, 6))
    vbar = unit(rng.standard_normal(6))
    st, err = oracle.compress_dense(S, vbar, 6)
    assert err < 1e-12
    assert oracle.rel_fro(oracle.materialize(st), S) < 1e-13


# ----------------------------------------------------------------------------
# recompression
# ----------------------------------------------------------------------------

def _factored_from_construction(d_k, d_v, sigma, rng, variant='gdn', mix=True):
    """Factors whose product is X diag(sigma) Y^T, hidden behind an invertible mixing G."""
    n = len(sigma)
    X = householder_orthogonal(d_k, rng)[:, :n]
    Y = householder_orthogonal(d_v, rng)[:, :n]
    G = np.eye(n) + (0.3 * rng.standard_normal((n, n)) if mix else 0)
    Ue = (X * sigma) @ G
    W = Y @ np.linalg.inv(G).T
    vbar = unit(rng.standard_normal(d_v))
    a = rng.standard_normal(d_k)
    if variant == 'kda':
        D = 0.5 + rng.random(d_k)
        st = oracle.FactoredState(a=a, U=Ue / D[:, None], W=W, vbar=vbar, D=D)
    else:
        c = 0.5 + rng.random(n)
        st = oracle.FactoredState(a=a, U=Ue / c[None, :], W=W, vbar=vbar, scale=c)
    return st, X, Y


@pytest.mark.parametrize('variant', ['gdn', 'kda'])
@pytest.mark.parametrize('r', [2, 4])
def test_recompress_constructed(variant, r):
    rng = np.random.default_rng(20 + r)
    sigma = np.array([6.0, 5.0, 3.0, 2.0, 1.0, 0.5])
    st, X, Y = _factored_from_construction(14, 11, sigma, rng, variant)
    new, err = oracle.recompress(st, r)
    expect = np.outer(st.a, st.vbar) + (X[:, :r] * sigma[:r]) @ Y[:, :r].T
    assert oracle.rel_fro(oracle.materialize(new), expect) < 1e-11
    assert err == pytest.approx(math.sqrt(np.sum(sigma[r:] ** 2)), rel=1e-10)
    assert new.m == r and np.array_equal(new.a, st.a)


def test_recompress_full_rank_is_identity():
    rng = np.random.default_rng(6)
    st, _, _ = _factored_from_construction(10, 9, np.array([3.0, 2.0, 1.0, 0.1]), rng)
    new, err = oracle.recompress(st, 4)
    assert err < 1e-12
    assert oracle.rel_fro(oracle.materialize(new), oracle.materialize(st)) < 1e-13


def test_recompress_matches_dense_truncation():
    # Eckart-Young by another route: SVD of the dense content U_eff W^T itself.
    rng = np.random.default_rng(7)
    d_k, d_v, m, r = 20, 16, 9, 4
    st = oracle.FactoredState(a=rng.standard_normal(d_k), U=rng.standard_normal((d_k, m)),
                              W=rng.standard_normal((d_v, m)), vbar=unit(rng.standard_normal(d_v)),
                              scale=0.2 + rng.random(m))
    M = st.U_eff() @ st.W.T
    new, err = oracle.recompress(st, r)
    s = np.linalg.svd(M, compute_uv=False)
    assert err == pytest.approx(math.sqrt(np.sum(s[r:] ** 2)), rel=1e-10)
    assert np.linalg.norm(M - new.U_eff() @ new.W.T) == pytest.approx(err, rel=1e-10)


def test_recompress_brute_force_optimality_tiny():
    # No rank-r matrix near the answer, nor any random one, does better (tiny head).
    rng = np.random.default_rng(8)
    d_k, d_v, m, r = 5, 4, 4, 2
    st = oracle.FactoredState(a=np.zeros(d_k), U=rng.standard_normal((d_k, m)),
                              W=rng.standard_normal((d_v, m)), vbar=unit(rng.standard_normal(d_v)),
                              scale=np.ones(m))
    M = st.U @ st.W.T
    new, err = oracle.recompress(st, r)
    U0, W0 = new.U, new.W
    for _ in range(3000):
        dU = 1e-3 * rng.standard_normal(U0.shape)
        dW = 1e-3 * rng.standard_normal(W0.shape)
        assert np.linalg.norm(M - (U0 + dU) @ (W0 + dW).T) >= err - 1e-12
        B = rng.standard_normal((d_k, r)) @ rng.standard_normal((r, d_v))
        assert np.linalg.norm(M - B) >= err


# ----------------------------------------------------------------------------
# Corollary 4: open-loop error across repeated compressions
# ----------------------------------------------------------------------------

def _gate_norm_bound(variant, tok, A):
    """Largest decay of one step: |Phi_t|_2 <= max gate (|I - beta k k^T|_2 = 1 for beta in [0, 1])."""
    if variant == 'gdn':
        return float(tok['alpha'])
    if variant == 'kda':
        return float(np.max(tok['alpha']))
    return math.exp(float(tok['dt']) * A)


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_open_loop_error_bounded_corollary4(variant):
    w = _small_workload(variant).with_(steps=120, T=6, rank=3)
    h = 2
    d = synth.head_dir(w, h)
    vbar = synth.sink_directions(w, [d])[0]
    A = float(synth.mamba2_A(w, [d])[0]) if variant == 'mamba2' else None
    S = oracle.dense_prefill(variant, synth.prefill_inputs(w, h), w.d_k, w.d_v, A)
    st, e = oracle.compress_dense(S, vbar, w.rank, variant)
    errs, taus = [e], [0]
    S_ref = S.copy()
    per_traj = e                       # sum_j eps_j prod_{s in (tau_j, t]} g_s, updated recursively
    g_bar = 0.0
    seen = []
    for t in range(1, w.steps + 1):
        tok = {kk: vv[0] for kk, vv in synth.token_inputs(w, synth.PHASE_DECODE, t - 1, [h]).items()}
        g_t = _gate_norm_bound(variant, tok, A)
        g_bar = max(g_bar, g_t)
        st, _ = oracle.factored_step(variant, st, tok, A)
        S_ref, _ = oracle.dense_step(variant, S_ref, tok, A)
        per_traj *= g_t
        dev = np.linalg.norm(oracle.materialize(st) - S_ref)
        assert dev <= per_traj * (1 + 1e-9) + 1e-12
        seen.append(dev)
        if t % w.T == 0:
            st, e = oracle.recompress(st, w.rank)
            errs.append(e)
            taus.append(t)
            per_traj += e
            dev = np.linalg.norm(oracle.materialize(st) - S_ref)
            assert dev <= per_traj * (1 + 1e-9) + 1e-12
            seen.append(dev)
    bound = oracle.open_loop_bound(max(errs), g_bar, w.T)
    assert max(seen) <= bound
    assert len(errs) == w.steps // w.T + 1
    # errors do not grow with the number of compressions (20 of them here)
    half = len(seen) // 2
    assert max(seen[half:]) <= bound


def test_open_loop_bound_formula():
    assert oracle.open_loop_bound(1.0, 0.5, 1) == pytest.approx(2.0)
    assert oracle.open_loop_bound(0.3, 0.9, 16) <= oracle.open_loop_bound(0.3, 0.9, 1)


# ----------------------------------------------------------------------------
# state bytes: the pages' Table 2 numbers
# ----------------------------------------------------------------------------

def test_state_bytes_reproduce_table2():
    with open(os.path.join(GOLDEN, 'state_bytes_table2.json')) as f:
        g = json.load(f)
    for model, p in g['printed'].items():
        inf = g['inferred'][model]
        H, dk, dv, R, Wi = inf['heads'], inf['d_k'], inf['d_v'], inf['R'], inf['interval']
        MB = lambda m: H * oracle.state_bytes(dk, dv, m, 4) / 1e6
        dense = H * oracle.dense_state_bytes(dk, dv, 4) / 1e6
        assert round(dense, 1) == p['orig_MB'], model
        assert round(MB(R), 1) == p['at_R_MB'], model
        assert round(MB(R + Wi / 2), 1) == p['mean_MB'], model
        assert round(MB(R + Wi), 1) == p['peak_MB'], model
        assert round(100 * MB(R) / dense) == p['bytes_pct'], model
        attn = 8192 * p['attn_B_per_token'] / 1e6
        assert round(dense + attn) == p['resident_orig_MB'], model
        assert round(MB(R + Wi / 2) + attn) == p['resident_seed_MB'], model


def test_state_bytes_halve_at_16_bit():
    assert oracle.state_bytes(128, 128, 40, 2) * 2 == oracle.state_bytes(128, 128, 40, 4)
