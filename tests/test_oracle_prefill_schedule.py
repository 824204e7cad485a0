"""Pins of the oracle's dense prefill and of the decode schedule in run_head.

The dense prefill is the plain recurrence over the prompt from S = 0
("Shallow Encoding Emits Deep Memories", picx.dev summary, Lemma 1, which
grows the state from S_0 = 0; thelatestinai.com list view, Table 1: the states
that leave the prefill are compressed at its end).  The decode schedule reads
out and updates every step and compresses back to rank r after every T-th step
(list view, Table 1, decode column); the output of step t is the read-out of the
state before that step's recompression.

Each test checks the oracle against an answer fixed by something else: a sum
written in closed form, a case worked by hand, the rank the schedule implies,
or the dense recurrence when nothing is truncated.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def unit(x):
    return x / np.linalg.norm(x)


def _gdn_tokens(K, V, alpha, beta, Q=None):
    L = len(K)
    return {'q': np.zeros_like(K) if Q is None else Q, 'k': K, 'v': V,
            'alpha': np.full(L, alpha) if np.isscalar(alpha) else np.asarray(alpha),
            'beta': np.full(L, beta) if np.isscalar(beta) else np.asarray(beta)}


# ----------------------------------------------------------------------------
# dense prefill
# ----------------------------------------------------------------------------

def test_prefill_orthonormal_keys_is_sum_of_outer_products():
    # alpha = beta = 1 and orthonormal keys: every erase sees k_t^T S = 0, so the
    # prefill from S = 0 stores each value at its key: S = sum_t k_t v_t^T = K^T V.
    rng = np.random.default_rng(10)
    d_k, d_v, L = 12, 9, 7
    Q, _ = np.linalg.qr(rng.standard_normal((d_k, d_k)))
    K = Q[:, :L].T.copy()                       # L orthonormal keys, one per row
    V = rng.standard_normal((L, d_v))
    S = oracle.dense_prefill('gdn', _gdn_tokens(K, V, 1.0, 1.0), d_k, d_v)
    assert np.allclose(S, K.T @ V, atol=1e-13)
    # the same keys under the per-channel gate with all channels at one
    tok = _gdn_tokens(K, V, 1.0, 1.0)
    tok['alpha'] = np.ones((L, d_k))
    S = oracle.dense_prefill('kda', tok, d_k, d_v)
    assert np.allclose(S, K.T @ V, atol=1e-13)


def test_prefill_gdn_three_tokens_by_hand():
    # d_k = d_v = 2, from S = 0, alpha = 1/2, beta = 1/2:
    # t0: k = e0, v = (2, 4):  S = beta k v^T            = [[1, 2], [0, 0]]
    # t1: k = e1, v = (6, 2):  S = alpha S + beta e1 v^T = [[0.5, 1], [3, 1]]
    # t2: k = e0, v = (0, 8):  erase: S - beta e0 (e0^T S) = [[0.25, 0.5], [3, 1]];
    #                          times alpha: [[0.125, 0.25], [1.5, 0.5]]; plus beta e0 v^T
    #                          = [[0, 4], [0, 0]]  ->  [[0.125, 4.25], [1.5, 0.5]]
    K = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0]])
    V = np.array([[2.0, 4.0], [6.0, 2.0], [0.0, 8.0]])
    S = oracle.dense_prefill('gdn', _gdn_tokens(K, V, 0.5, 0.5), 2, 2)
    assert np.allclose(S, [[0.125, 4.25], [1.5, 0.5]], atol=0, rtol=1e-15)


def test_prefill_mamba2_is_the_decayed_cumulative_sum():
    # S_L = exp(A sum dt) S0 + sum_t exp(A sum_{s>t} dt_s) dt_t B_t x_t^T, summed here
    # term by term (no recursion), from a nonzero S0.
    rng = np.random.default_rng(11)
    d_k, d_v, L, A = 10, 6, 9, -1.7
    S0 = rng.standard_normal((d_k, d_v))
    B = rng.standard_normal((L, d_k))
    X = rng.standard_normal((L, d_v))
    dt = rng.uniform(0.05, 0.6, L)
    tok = {'C': np.zeros((L, d_k)), 'B': B, 'x': X, 'dt': dt}
    S = oracle.dense_prefill('mamba2', tok, d_k, d_v, A=A, S0=S0)
    ref = math.exp(A * dt.sum()) * S0
    for t in range(L):
        ref = ref + math.exp(A * dt[t + 1:].sum()) * dt[t] * np.outer(B[t], X[t])
    assert np.allclose(S, ref, atol=1e-13)
    # from S = 0 the first term goes
    S = oracle.dense_prefill('mamba2', tok, d_k, d_v, A=A)
    assert np.allclose(S, ref - math.exp(A * dt.sum()) * S0, atol=1e-13)


def test_prefill_from_nonzero_state_with_no_writes_only_decays():
    # beta = 0: S_L = (prod alpha_t) S0 for the scalar gate, diag(prod alpha_t) S0 per channel
    rng = np.random.default_rng(12)
    d_k, d_v, L = 8, 5, 6
    S0 = rng.standard_normal((d_k, d_v))
    K = np.array([unit(rng.standard_normal(d_k)) for _ in range(L)])
    V = rng.standard_normal((L, d_v))
    alpha = rng.uniform(0.8, 1.0, L)
    S = oracle.dense_prefill('gdn', _gdn_tokens(K, V, alpha, 0.0), d_k, d_v, S0=S0)
    assert np.allclose(S, np.prod(alpha) * S0, atol=1e-14)
    tok = _gdn_tokens(K, V, 1.0, 0.0)
    tok['alpha'] = rng.uniform(0.8, 1.0, (L, d_k))
    S = oracle.dense_prefill('kda', tok, d_k, d_v, S0=S0)
    assert np.allclose(S, np.prod(tok['alpha'], axis=0)[:, None] * S0, atol=1e-14)


def test_prefill_starts_from_zero_and_uses_every_token():
    # one token from S = 0 with beta = 1 stores exactly k v^T (no leftover S0, none dropped);
    # the order of two writes at the same unit key decides which value stays
    k = np.array([0.0, 1.0, 0.0])
    v1, v2 = np.array([1.0, -2.0]), np.array([3.0, 5.0])
    S = oracle.dense_prefill('gdn', _gdn_tokens(k[None], v1[None], 0.9, 1.0), 3, 2)
    assert np.allclose(S, np.outer(k, v1), atol=0)
    S = oracle.dense_prefill('gdn', _gdn_tokens(np.array([k, k]), np.array([v1, v2]), 1.0, 1.0), 3, 2)
    assert np.allclose(S, np.outer(k, v2), atol=1e-15)


# ----------------------------------------------------------------------------
# decode schedule (run_head)
# ----------------------------------------------------------------------------

def _head(variant, d_k=16, d_v=12, steps=24):
    base = {'gdn': synth.GDN_BATCHED, 'kda': synth.KDA_BATCHED, 'mamba2': synth.MAMBA2_BATCHED}[variant]
    w = base.with_(n_req=1, n_head=2, d_k=d_k, d_v=d_v, rank=3, T=4, steps=steps, prefill_len=20)
    h = 1
    d = synth.head_dir(w, h)
    vbar = synth.sink_directions(w, [d])[0]
    A = float(synth.mamba2_A(w, [d])[0]) if variant == 'mamba2' else None
    S = oracle.dense_prefill(variant, synth.prefill_inputs(w, h), d_k, d_v, A)

    def tokens(t):
        return {kk: vv[0] for kk, vv in synth.token_inputs(w, synth.PHASE_DECODE, t, [h]).items()}
    return w, vbar, A, S, tokens


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_run_head_without_truncation_follows_the_dense_recurrence(variant):
    # r >= min(d_k, d_v) keeps every singular value, so compressions change nothing and
    # the outputs are those of the dense recurrence from the prefill state, token 0 first
    w, vbar, A, S, tokens = _head(variant)
    traj = oracle.run_head(variant, S, vbar, r=max(w.d_k, w.d_v), T=2, step_tokens=tokens,
                           steps=w.steps, A=A, compress=True)
    S_ref = S.copy()
    for t in range(w.steps):
        S_ref, o_ref = oracle.dense_step(variant, S_ref, tokens(t), A)
        assert oracle.rel_fro(traj.outputs[t], o_ref) < 1e-10, t
    assert oracle.rel_fro(oracle.materialize(traj.final), S_ref) < 1e-10


@pytest.mark.parametrize('T,steps', [(2, 10), (3, 12), (5, 12)])
def test_run_head_compression_count(T, steps):
    w, vbar, A, S, tokens = _head('gdn', steps=steps)
    traj = oracle.run_head('gdn', S, vbar, r=3, T=T, step_tokens=tokens, steps=steps)
    assert len(traj.compress_errors) == steps // T + 1
    assert len(traj.outputs) == steps


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_run_head_content_rank_follows_the_schedule(variant):
    # after compress_dense the content has rank r; each step writes one new value
    # direction eps (the erase term lies in the old row space, and KDA's second column
    # pairs with a W column in span(W)), so the content rank grows by one a step; a
    # recompression after step t (T | t) brings it back to r.  The recorded state of
    # step t is taken before that step's recompression, so its content rank is
    # r + ((t - 1) mod T) + 1, and the final state (after the last recompression,
    # steps a multiple of T) has rank r.
    w, vbar, A, S, tokens = _head(variant, d_k=24, d_v=20)
    r, T, steps = 2, 3, 12
    rec = list(range(1, steps + 1))
    traj = oracle.run_head(variant, S, vbar, r=r, T=T, step_tokens=tokens, steps=steps, A=A,
                           record_states=rec)

    def content_rank(St):
        C = St - np.outer(St @ vbar / (vbar @ vbar), vbar)
        s = np.linalg.svd(C, compute_uv=False)
        return int(np.sum(s > 1e-9 * s[0]))
    for t in rec:
        assert content_rank(traj.states[t]) == r + ((t - 1) % T) + 1, t
    assert content_rank(oracle.materialize(traj.final)) == r


@pytest.mark.parametrize('variant', ['gdn', 'mamba2'])
def test_run_head_output_reads_the_state_before_recompression(variant):
    # o_T = S_T^T q_T with S_T the uncompressed state of step T; the read-out of the
    # recompressed state differs (the truncation discards content), so the test sees
    # a recompression moved before the read-out
    w, vbar, A, S, tokens = _head(variant)
    T = 4
    traj = oracle.run_head(variant, S, vbar, r=2, T=T, step_tokens=tokens, steps=2 * T, A=A,
                           record_states=[T, T + 1])
    qname = 'C' if variant == 'mamba2' else 'q'
    q_T = tokens(T - 1)[qname]
    o_before = traj.states[T].T @ q_T
    assert np.allclose(traj.outputs[T - 1], o_before, atol=1e-12 * np.linalg.norm(o_before))
    # the state after the recompression of step T, stepped once, is what step T+1 reads
    S_trunc = traj.states[T + 1]
    o_next = S_trunc.T @ tokens(T)[qname]
    assert np.allclose(traj.outputs[T], o_next, atol=1e-12 * np.linalg.norm(o_next))
    # and the recompression changed the state: its read-out at q_T differs from o_T
    st_T, _ = oracle.compress_dense(S, vbar, 2, variant)
    for t in range(T):
        st_T, _ = oracle.factored_step(variant, st_T, tokens(t), A)
    st_c, err = oracle.recompress(st_T, 2)
    assert err > 0
    o_after = oracle.materialize(st_c).T @ q_T
    assert np.linalg.norm(o_after - o_before) > 1e-6 * np.linalg.norm(o_before)
