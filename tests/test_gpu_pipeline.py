"""End-to-end parity on the five synthetic workloads at full size (needs a GPU).

The GPU runs every head of the workload the way the benchmark does: dense
prefill with in-kernel prompt tokens, compression to rank r, then the decode
loop with recompression every T steps.  The oracle runs sampled heads from
the host twin of the generator (its own prefill, compression and decode), and
the two are compared as reconstructed states and read-outs.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import rank_state_compression_head_b300 as R
import synth
from _gpu import TOL, normwise_out_err, rel_err
from rank_state_compression_head_b300.workload import DeviceRun

pytestmark = pytest.mark.gpu


def head_view(buf, h: int) -> R.seed_state:
    """A seed_state covering head h alone (pointer offsets into the same buffers)."""
    st = buf.st
    v = R.seed_state()
    ctypes.memmove(ctypes.byref(v), ctypes.byref(st), ctypes.sizeof(st))
    v.n_heads = 1
    v.head_order = None  # the class order lists all heads; a one-head view has none
    v.a = st.a + h * buf.d_k * 4
    v.status = st.status + h * 4
    if st.vbar_index:
        v.vbar_index = st.vbar_index + h * 4
    if st.rank:
        v.rank = st.rank + h * 4
        v.col_offset = st.col_offset + h * 8
    else:
        esz = buf.U.element_size()
        v.U = st.U + h * buf.cap * buf.d_k * esz
        v.W = st.W + h * buf.cap * buf.d_v * esz
        if buf.variant != 'kda':
            v.scale = st.scale + h * buf.cap * 4
    if buf.variant == 'kda':
        v.scale = st.scale + h * buf.d_k * 4
    return v


def gpu_head_states(buf, heads):
    out = torch.empty(len(heads), buf.d_k, buf.d_v, device='cuda')
    for i, h in enumerate(heads):
        R.seed_materialize(head_view(buf, int(h)), out[i])
    return out


def oracle_head(w, h, steps, record, compress=True):
    d = synth.head_dir(w, h)
    vbar = synth.sink_directions(w, [d])[0]
    A = float(synth.mamba2_A(w, [d])[0]) if w.variant == 'mamba2' else None
    r = int(synth.head_ranks(w, [h])[0])
    L = int(synth.prompt_lengths(w, [h // w.n_dir])[0])
    S0 = oracle.dense_prefill(w.variant, synth.prefill_inputs(w, h, L), w.d_k, w.d_v, A)

    def tok(t):
        return {k: v[0] for k, v in synth.decode_inputs(w, t, [h]).items()}

    return oracle.run_head(w.variant, S0, vbar, r, w.T, tok, steps, A, record_states=record,
                           compress=compress), tok, A


def run_pipeline(w, sample, steps, record):
    run = DeviceRun(w)
    S = run.prefill()
    err0 = torch.zeros(run.H, device='cuda')
    run.compress(S, err0)
    idx = torch.tensor(sample, device='cuda')
    outs = torch.empty(steps, len(sample), w.d_v, device='cuda')
    states = {}
    for t in range(1, steps + 1):
        run.gen_inputs(t - 1)
        run.decode()
        outs[t - 1] = run.o[idx]
        if t in record:
            states[t] = gpu_head_states(run.state, sample)
        if t % w.T == 0:
            run.recompress(run.trunc)
            bad = int((run.state.status[:run.H] != 0).sum())
            assert bad == 0, f'recompress status after step {t}: {bad} heads'
    torch.cuda.synchronize()
    status = run.state.status[:run.H]
    assert int((status != 0).sum()) == 0, 'device status'
    final = gpu_head_states(run.state, sample)
    return run, S, outs.double().cpu().numpy(), {t: s.double().cpu().numpy() for t, s in states.items()}, \
        final.double().cpu().numpy(), err0[idx].double().cpu().numpy()


def sample_heads(w, n):
    rng = np.random.default_rng(w.seed + 1000)
    heads = sorted(set(rng.choice(w.n_heads, size=n, replace=False).tolist()) | {0, w.n_heads - 1})
    return heads


CASES = {
    'gdn_tiny_b1_h4_r8': dict(n=4, steps=None),
    'gdn_batched_b64_h32_r32': dict(n=6, steps=None),
    'kda_batched_b128_h32_r32': dict(n=4, steps=None),
    'mamba2_batched_b256_h128_r16': dict(n=5, steps=None),
    'gdn_serving_b512_l36_h32_ragged': dict(n=4, steps=None),
}


@pytest.mark.parametrize('name', list(CASES))
def test_workload_matches_oracle(name, record_property):
    w = synth.WORKLOADS[name]
    steps = CASES[name]['steps'] or w.steps
    sample = sample_heads(w, CASES[name]['n']) if w.n_heads > 4 else list(range(w.n_heads))
    record = sorted({1, w.T - 1, w.T + 3, steps // 2 + 1, steps - 1} - {0})
    record = [t for t in record if t % w.T != 0]
    run, S_gpu, outs, states, final, err0 = run_pipeline(w, sample, steps, record)
    tol = TOL[w.factor_dtype]
    worst = dict(state=0.0, out=0.0, pooled=0.0, final=0.0)
    every = list(range(1, steps + 1))
    for i, h in enumerate(sample):
        # the oracle's state at every step: the normwise read-out error is checked at each one
        traj, tok, A = oracle_head(w, h, steps, every)
        for t in record:
            worst['state'] = max(worst['state'], rel_err(states[t][i], traj.states[t]))
        ref_final = oracle.materialize(traj.final)
        worst['final'] = max(worst['final'], rel_err(final[i], ref_final))
        o_ref = np.array(traj.outputs)
        worst['pooled'] = max(worst['pooled'], rel_err(outs[:, i], o_ref))
        # normwise read-out error at every step (state norm of the oracle there)
        for t in every:
            q = tok(t - 1)['C' if w.variant == 'mamba2' else 'q']
            worst['out'] = max(worst['out'], normwise_out_err(outs[t - 1, i], o_ref[t - 1], traj.states[t], q))
        # truncation error of the end-of-prefill compression, up to fp32 rounding of the state
        e_ref = traj.compress_errors[0]
        assert abs(err0[i] - e_ref) <= tol * e_ref + 1e-5 * np.linalg.norm(traj.prefill_state), h
    record_property('parity', dict(case=name, tol=tol, heads=len(sample), steps=steps, **worst))
    print(name, {k: f'{v:.2e}' for k, v in worst.items()})
    assert max(worst.values()) < tol, worst


def test_tiny_factored_without_compression_equals_dense():
    """Within one interval the factored trajectory is the dense recurrence (no truncation)."""
    w = synth.GDN_TINY
    run = DeviceRun(w)
    S = run.prefill()
    run.compress(S)
    heads = list(range(w.n_heads))
    outs = []
    for t in range(w.T):
        run.gen_inputs(t)
        run.decode()
        outs.append(run.o.double().cpu().numpy().copy())
    states = gpu_head_states(run.state, heads).double().cpu().numpy()
    for h in heads:
        traj, tok, _ = oracle_head(w, h, 0, [])
        st0, _ = oracle.compress_dense(traj.prefill_state, synth.sink_directions(w, [h])[0], w.rank)
        Sd = oracle.materialize(st0)
        for t in range(w.T):
            Sd, o = oracle.gdn_dense_step(Sd, **{k: v for k, v in tok(t).items()})
            assert rel_err(outs[t][h], o) < TOL['f32']
        assert rel_err(states[h], Sd) < TOL['f32']


@pytest.mark.parametrize('name', ['gdn_batched_b64_h32_r32', 'kda_batched_b128_h32_r32',
                                  'mamba2_batched_b256_h128_r16'])
def test_dense_comparator_full_size(name):
    """The dense-state kernel on the full workload, sampled heads against the oracle recurrence."""
    w = synth.WORKLOADS[name]
    run = DeviceRun(w)
    S = run.prefill()
    sample = sample_heads(w, 3)
    idx = torch.tensor(sample, device='cuda')
    n = 5
    outs = []
    for t in range(n):
        run.gen_inputs(t)
        run.dense_step(S)
        outs.append(run.o[idx].double().cpu().numpy())
    Sg = S[idx].double().cpu().numpy()
    for i, h in enumerate(sample):
        traj, tok, A = oracle_head(w, h, 0, [])
        Sd = traj.prefill_state
        for t in range(n):
            Sd, o = oracle.dense_step(w.variant, Sd, tok(t), A)
            assert rel_err(outs[t][i], o) < 1e-4
        assert rel_err(Sg[i], Sd) < 1e-4
