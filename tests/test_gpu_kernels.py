"""Per-call parity of the CUDA kernels against the CPU oracle (needs a GPU).

Small head counts with ragged ranks (several column tiles and ragged tails),
inputs from the seeded generator, the same stored values on both sides.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_state_compression_head_b300 as R
import synth
from _gpu import (TOL, gpu_dense, make_buffers, normwise_out_err, random_states, rel_err, stored,
                  to_dev, upload)

pytestmark = pytest.mark.gpu

D_V = {'gdn': 128, 'kda': 128, 'mamba2': 64}
BASE = {'gdn': synth.GDN_BATCHED, 'kda': synth.KDA_BATCHED, 'mamba2': synth.MAMBA2_BATCHED}


def ranks_for(variant, H, T):
    growth = 2 if variant == 'kda' else 1
    top = 64 - growth * T
    base = [1, 7, top, 16, 31, 5, top - 1, 24]
    return np.array([base[h % len(base)] for h in range(H)], dtype=np.int32)


def inputs(variant, t, H, seed_shift=0):
    w = BASE[variant].with_(seed=BASE[variant].seed + 100 + seed_shift, n_req=1, n_layers=1, n_head=H)
    d = synth.token_inputs(w, synth.PHASE_DECODE, t, np.arange(H))
    return d


def dev_inputs(variant, d):
    if variant == 'mamba2':
        return dict(q=to_dev(d['C']), k=to_dev(d['B']), v=to_dev(d['x']), gate=to_dev(d['dt']), beta=None)
    return dict(q=to_dev(d['q']), k=to_dev(d['k']), v=to_dev(d['v']), gate=to_dev(d['alpha']),
                beta=to_dev(d['beta']))


def head_tok(d, h):
    return {k: v[h] for k, v in d.items()}


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
@pytest.mark.parametrize('dtype', ['f32', 'bf16', 'f16'])
def test_materialize_matches_oracle(variant, dtype):
    H, T, s = 13, 8, 3
    ranks = ranks_for(variant, H, T)
    states, vbar = random_states(11, H, 128, D_V[variant], ranks, s, T, variant, dtype)
    buf = make_buffers(variant, dtype, H, 128, D_V[variant], T, vbar, ranks)
    upload(buf, states, s)
    S = gpu_dense(buf)
    for h in range(H):
        assert rel_err(S[h], oracle.materialize(states[h])) < 1e-5


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
@pytest.mark.parametrize('dtype', ['f32', 'bf16', 'f16'])
def test_decode_steps_match_oracle(variant, dtype):
    H, T, s0 = 37, 8, 2
    ranks = ranks_for(variant, H, T)
    states, vbar = random_states(12, H, 128, D_V[variant], ranks, s0, T, variant, dtype)
    buf = make_buffers(variant, dtype, H, 128, D_V[variant], T, vbar, ranks)
    upload(buf, states, s0)
    A = -(1.0 + 15.0 * synth.uniforms(5, 0, 99, 0, np.arange(H), 1)[:, 0]).astype(np.float32).astype(np.float64)
    A_dev = to_dev(A) if variant == 'mamba2' else None
    o = torch.empty(H, D_V[variant], device='cuda')
    worst_o, pooled = 0.0, 0.0
    for t in range(s0, T):
        d = inputs(variant, t, H)
        di = dev_inputs(variant, d)
        R.seed_decode_step(buf.st, di['q'], di['k'], di['v'], di['gate'], di['beta'], A_dev, o)
        torch.cuda.synchronize()
        o_gpu = o.double().cpu().numpy()
        o_ref = np.zeros_like(o_gpu)
        for h in range(H):
            states[h], o_ref[h] = oracle.factored_step(variant, states[h], head_tok(d, h), A[h])
            qv = d['C'][h] if variant == 'mamba2' else d['q'][h]
            worst_o = max(worst_o, normwise_out_err(o_gpu[h], o_ref[h], oracle.materialize(states[h]), qv))
        pooled = max(pooled, rel_err(o_gpu, o_ref))
    assert buf.st.steps_since_compress == T
    assert int(buf.status.abs().sum()) == 0
    S = gpu_dense(buf)
    worst_s = max(rel_err(S[h], oracle.materialize(states[h])) for h in range(H))
    print(f'{variant} {dtype}: state {worst_s:.2e} out normwise {worst_o:.2e} pooled {pooled:.2e}')
    assert worst_s < TOL[dtype] and worst_o < TOL[dtype] and pooled < TOL[dtype]
    with pytest.raises(R.SeedError) as e:
        R.seed_decode_step(buf.st, di['q'], di['k'], di['v'], di['gate'], di['beta'], A_dev, o)
    assert e.value.status == R.SEED_ERR_CAPACITY


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
@pytest.mark.parametrize('dtype', ['f32', 'bf16', 'f16'])
def test_recompress_matches_oracle(variant, dtype):
    H, T = 21, 8
    growth = 2 if variant == 'kda' else 1
    ranks = ranks_for(variant, H, T)
    states, vbar = random_states(13, H, 128, D_V[variant], ranks, T, T, variant, dtype)
    buf = make_buffers(variant, dtype, H, 128, D_V[variant], T, vbar, ranks)
    upload(buf, states, T)
    err = torch.zeros(H, device='cuda')
    R.seed_recompress(buf.st, err)
    torch.cuda.synchronize()
    assert buf.st.steps_since_compress == 0
    assert int(buf.status.abs().sum()) == 0
    S = gpu_dense(buf)
    err = err.double().cpu().numpy()
    for h in range(H):
        ref, e_ref = oracle.recompress(states[h], int(ranks[h]))
        S_ref = oracle.materialize(ref)
        assert rel_err(S[h], S_ref) < TOL[dtype], h
        assert abs(err[h] - e_ref) <= TOL[dtype] * max(e_ref, 1e-3 * np.linalg.norm(S_ref)), h
        assert ref.m == ranks[h]


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
@pytest.mark.parametrize('dtype', ['f32', 'bf16', 'f16'])
def test_compress_dense_matches_oracle(variant, dtype):
    H, T, d_v = 9, 8, D_V[variant]
    ranks = ranks_for(variant, H, T)
    rng = np.random.default_rng(14)
    vbar = rng.standard_normal((H, d_v))
    vbar = stored(vbar / np.linalg.norm(vbar, axis=1, keepdims=True), 'f32')
    # states with a sink along vbar and a decaying spectrum
    S = np.zeros((H, 128, d_v))
    for h in range(H):
        X = rng.standard_normal((128, d_v)) * (0.97 ** np.arange(d_v))[None, :]
        S[h] = 3.0 * np.outer(rng.standard_normal(128), vbar[h]) + X @ rng.standard_normal((d_v, d_v)) / np.sqrt(d_v)
    S = stored(S, 'f32')
    buf = make_buffers(variant, dtype, H, 128, d_v, T, vbar, ranks)
    buf.st.steps_since_compress = 5
    err = torch.zeros(H, device='cuda')
    R.seed_compress_dense(to_dev(S), buf.st, err)
    torch.cuda.synchronize()
    assert buf.st.steps_since_compress == 0
    assert int(buf.status.abs().sum()) == 0
    Sg = gpu_dense(buf)
    err = err.double().cpu().numpy()
    for h in range(H):
        ref, e_ref = oracle.compress_dense(S[h], vbar[h], int(ranks[h]), variant)
        assert np.allclose(buf.a[h].double().cpu().numpy(), ref.a, rtol=1e-5, atol=1e-5 * np.abs(ref.a).max())
        assert rel_err(Sg[h], oracle.materialize(ref)) < TOL[dtype], h
        assert abs(err[h] - e_ref) <= TOL[dtype] * e_ref, h


@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_dense_decode_step_matches_oracle(variant):
    H, d_v = 19, D_V[variant]
    rng = np.random.default_rng(15)
    S = stored(rng.standard_normal((H, 128, d_v)), 'f32')
    A = stored(-(1 + 15 * rng.random(H)), 'f32')
    S_dev = to_dev(S)
    o = torch.empty(H, d_v, device='cuda')
    for t in range(3):
        d = inputs(variant, t, H, seed_shift=7)
        di = dev_inputs(variant, d)
        R.seed_dense_decode_step(R.VARIANTS[variant], H, 128, d_v, S_dev, di['q'], di['k'], di['v'],
                                 di['gate'], di['beta'], to_dev(A) if variant == 'mamba2' else None,
                                 None, o)
        torch.cuda.synchronize()
        o_ref = np.zeros((H, d_v))
        for h in range(H):
            S[h], o_ref[h] = oracle.dense_step(variant, S[h], head_tok(d, h), A[h])
        assert rel_err(S_dev.double().cpu().numpy(), S) < 1e-5
        assert rel_err(o.double().cpu().numpy(), o_ref) < 1e-5


def test_zero_heads_and_nonfinite_status():
    H, T, s = 6, 8, 1
    ranks = ranks_for('gdn', H, T)
    states, vbar = random_states(16, H, 128, 128, ranks, s, T, 'gdn', 'bf16')
    buf = make_buffers('gdn', 'bf16', H, 128, 128, T, vbar, ranks)
    upload(buf, states, s)
    d = inputs('gdn', 0, H)
    d['q'] = d['q'].copy()
    d['q'][3, 5] = np.nan
    di = dev_inputs('gdn', d)
    o = torch.empty(H, 128, device='cuda')
    R.seed_decode_step(buf.st, di['q'], di['k'], di['v'], di['gate'], di['beta'], None, o)
    torch.cuda.synchronize()
    status = buf.status.cpu().numpy()
    assert status[3] == R.SEED_ERR_NONFINITE
    assert np.all(np.delete(status, 3) == 0)
    empty = make_buffers('gdn', 'bf16', 0, 128, 128, T, vbar[:1], ranks[:0])
    R.seed_decode_step(empty.st, None, None, None, None, None, None, None)
    R.seed_recompress(empty.st)
    assert empty.st.steps_since_compress == 0


@pytest.mark.parametrize('variant', ['gdn', 'mamba2'])
def test_rank_zero_sink_only(variant):
    # r = 0: the state is the sink alone after each compression
    H, T = 4, 4
    ranks = np.zeros(H, dtype=np.int32)
    states, vbar = random_states(17, H, 128, D_V[variant], ranks, 0, T, variant, 'f32')
    buf = make_buffers(variant, 'f32', H, 128, D_V[variant], T, vbar, ranks, ragged=False)
    upload(buf, states, 0)
    A = np.full(H, -2.0)
    o = torch.empty(H, D_V[variant], device='cuda')
    for t in range(T):
        d = inputs(variant, t, H)
        di = dev_inputs(variant, d)
        R.seed_decode_step(buf.st, di['q'], di['k'], di['v'], di['gate'], di['beta'],
                           to_dev(A) if variant == 'mamba2' else None, o)
        for h in range(H):
            states[h], _ = oracle.factored_step(variant, states[h], head_tok(d, h), A[h])
    R.seed_recompress(buf.st)
    S = gpu_dense(buf)
    for h in range(H):
        ref, _ = oracle.recompress(states[h], 0)
        assert rel_err(S[h], oracle.materialize(ref)) < 1e-4
