"""Device twin of the workload generator, and the dense prefill with in-kernel
prompt tokens, against the host generator and the oracle (needs a GPU)."""
import numpy as np
import pytest
import torch

import oracle
import rank_state_compression_head_b300 as R
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize('seed,phase,field,time,entity0', [
    (0, 0, 0, 0, 0), (1, 2, 1, 7, 100), (4, 1, 3, 8191, 589000), (0xFFFFFFFF, 2, 20, 3, 5)])
def test_raw_words_bit_exact(seed, phase, field, time, entity0):
    n_ent, n_blocks = 37, 33
    out = torch.zeros(n_ent * n_blocks * 4, dtype=torch.int32, device='cuda')
    R.seed_synth_raw(seed, phase, field, time, entity0, n_ent, n_blocks, out)
    dev = out.cpu().numpy().view(np.uint32).reshape(n_ent, 4 * n_blocks)
    host = synth.raw_words(seed, phase, field, time, entity0 + np.arange(n_ent), n_blocks)
    assert np.array_equal(dev, host)


def close(dev, host, rtol=2e-6):
    dev = np.asarray(dev, np.float64)
    return np.max(np.abs(dev - host) / (1.0 + np.abs(host))) < rtol


@pytest.mark.parametrize('name', list(synth.WORKLOADS))
def test_constants_and_step_inputs_match_host(name):
    w = synth.WORKLOADS[name]
    run_heads = min(w.n_heads, 300)
    wst = R.synth_workload_struct(w)
    vbar = torch.empty(w.n_dir, w.d_v, device='cuda')
    sink = torch.empty(w.n_dir, device='cuda')
    A = torch.empty(w.n_dir, device='cuda')
    ranks = torch.empty(w.n_heads, dtype=torch.int32, device='cuda')
    plen = torch.empty(w.n_req, dtype=torch.int32, device='cuda')
    R.seed_synth_constants(wst, vbar, sink, A, ranks, plen)
    torch.cuda.synchronize()
    assert close(vbar.cpu(), synth.sink_directions(w))
    assert close(sink.cpu(), synth.sink_scales(w))
    if w.variant == 'mamba2':
        assert close(A.cpu(), synth.mamba2_A(w))
    assert np.array_equal(ranks.cpu().numpy(), synth.head_ranks(w))
    assert np.array_equal(plen.cpu().numpy(), synth.prompt_lengths(w))
    head0 = w.n_heads - run_heads
    q = torch.empty(run_heads, w.d_k, device='cuda')
    k = torch.empty_like(q)
    v = torch.empty(run_heads, w.d_v, device='cuda')
    gate = torch.empty(run_heads, w.d_k, device='cuda') if w.variant == 'kda' else torch.empty(run_heads, device='cuda')
    beta = torch.empty(run_heads, device='cuda')
    for step in (0, w.steps - 1):
        R.seed_synth_step_inputs(wst, synth.PHASE_DECODE, step, head0, run_heads, vbar, sink, q, k, v, gate, beta)
        torch.cuda.synchronize()
        d = synth.decode_inputs(w, step, np.arange(head0, w.n_heads))
        if w.variant == 'mamba2':
            pairs = [(q, d['C']), (k, d['B']), (v, d['x']), (gate, d['dt'])]
        else:
            pairs = [(q, d['q']), (k, d['k']), (v, d['v']), (gate, d['alpha']), (beta, d['beta'])]
        for dev, host in pairs:
            assert close(dev.cpu(), host), name


def _prefill_vs_oracle(w, chunked, tol=1e-5):
    from rank_state_compression_head_b300.workload import DeviceRun
    run = DeviceRun(w)
    S = run.prefill(chunked=chunked)
    torch.cuda.synchronize()
    S = S.double().cpu().numpy()
    L = synth.prompt_lengths(w)
    worst = 0.0
    for h in range(w.n_heads):
        A = float(synth.mamba2_A(w, [synth.head_dir(w, h)])[0]) if w.variant == 'mamba2' else None
        toks = synth.prefill_inputs(w, h, int(L[h // w.n_dir]))
        ref = oracle.dense_prefill(w.variant, toks, w.d_k, w.d_v, A)
        err = np.linalg.norm(S[h] - ref) / np.linalg.norm(ref)
        assert err < tol, (h, err)
        worst = max(worst, err)
    return worst


_PREFILL_BASE = {'gdn': synth.GDN_TINY, 'kda': synth.KDA_BATCHED, 'mamba2': synth.MAMBA2_BATCHED}


@pytest.mark.parametrize('chunked', [False, True], ids=['serial', 'chunked'])
@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_dense_prefill_matches_oracle(variant, chunked):
    w = _PREFILL_BASE[variant].with_(n_req=3, n_head=4, prefill_len=0, prefill_range=(40, 90))
    _prefill_vs_oracle(w, chunked)


@pytest.mark.parametrize('L', [1, 15, 16, 17, 31, 32, 33, 64, 95])
@pytest.mark.parametrize('variant', ['gdn', 'kda', 'mamba2'])
def test_chunked_prefill_chunk_edges(variant, L):
    # prompt lengths on and around the 16- and 32-token chunk boundaries, both value widths
    for dv in (64, 128):
        w = _PREFILL_BASE[variant].with_(n_req=2, n_head=2, d_v=dv, prefill_len=L)
        _prefill_vs_oracle(w, True)


def test_chunked_prefill_mamba2_decay_underflow():
    # exp(dt A) products over a chunk fall far below fp32's range; the chunks carry their logarithm
    w = synth.MAMBA2_BATCHED.with_(n_req=2, n_head=3, prefill_len=70, a_range=(16.0, 16.0), dt_mu=1.0)
    _prefill_vs_oracle(w, True)


@pytest.mark.parametrize('alpha', [(0.3, 0.5), (0.02, 0.1)], ids=['steep', 'below_range'])
@pytest.mark.parametrize('variant', ['gdn', 'kda'])
def test_chunked_prefill_steep_gates(variant, alpha):
    # steep gates stay on the chunked kernel while alpha_lo^C >= 2^-96; below that the call
    # hands over to the token-serial kernel; both must give the recurrence's state
    w = _PREFILL_BASE[variant].with_(n_req=2, n_head=2, prefill_len=77, alpha_range=alpha)
    _prefill_vs_oracle(w, True)


def test_chunked_prefill_matches_serial_at_full_prompt():
    # serving-length prompts (up to 2048 tokens): the chunked and serial kernels agree state by state
    from rank_state_compression_head_b300.workload import DeviceRun
    for variant in ('gdn', 'kda', 'mamba2'):
        w = _PREFILL_BASE[variant].with_(n_req=4, n_head=8, prefill_len=0, prefill_range=(1500, 2048))
        run = DeviceRun(w)
        a = run.prefill(chunked=False)
        b = run.prefill(chunked=True)
        torch.cuda.synchronize()
        err = ((a - b).flatten(1).norm(dim=1) / a.flatten(1).norm(dim=1)).max().item()
        assert err < 1e-4, (variant, err)
        # and two heads against the oracle
        L = synth.prompt_lengths(w)
        for h in (0, w.n_heads - 1):
            A = float(synth.mamba2_A(w, [synth.head_dir(w, h)])[0]) if variant == 'mamba2' else None
            toks = synth.prefill_inputs(w, h, int(L[h // w.n_dir]))
            ref = oracle.dense_prefill(variant, toks, w.d_k, w.d_v, A)
            e = np.linalg.norm(b[h].double().cpu().numpy() - ref) / np.linalg.norm(ref)
            assert e < 1e-4, (variant, h, e)
