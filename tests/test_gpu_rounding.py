"""Storage formats and rounding of the 16-bit factors (needs a GPU).

"Shallow Encoding Emits Deep Memories", picx.dev summary, Practical
implications (fp16 factors) and thelatestinai.com list view, the drift table
by storage format and rounding (round to nearest and stochastic rounding).

* stochastic rounding is reproducible for a seed and changes with it;
* it is unbiased: over many copies of one value the stored copies take only the
  two neighbouring 16-bit values, and their mean is the value (checked against
  the same computation stored in fp32), while round-to-nearest picks the
  nearer neighbour;
* the drift of a decode trajectory against the float64 oracle, per storage
  format and rounding, stays within the 16-bit tolerance; the figures are
  printed in the run's parity block.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_state_compression_head_b300 as R
import synth
from _gpu import TOL, gpu_dense, make_buffers, random_states, rel_err, upload
from rank_state_compression_head_b300.workload import DeviceRun

pytestmark = pytest.mark.gpu

NEIGHBOURS = {'bf16': torch.bfloat16, 'f16': torch.float16}


def _append_copies(dtype, rounding, H, k, seed=7):
    """Decode one step on H empty (rank 0) heads with the same inputs: each head
    appends the key k as its first U column, rounded to the storage format."""
    T = 4
    vbar = np.zeros((H, 128))
    vbar[:, 0] = 1.0
    buf = make_buffers('gdn', dtype, H, 128, 128, T, vbar, np.zeros(H, np.int32), ragged=False,
                       rounding=rounding, sr_seed=seed)
    dev = lambda x: torch.tensor(np.asarray(x), dtype=torch.float32, device='cuda').contiguous()
    kk = dev(np.broadcast_to(k, (H, 128)))
    v = dev(np.ones((H, 128)))
    o = torch.empty(H, 128, device='cuda')
    R.seed_decode_step(buf.st, kk, kk, v, dev(np.full(H, 0.9)), dev(np.full(H, 0.5)), None, o)
    torch.cuda.synchronize()
    assert int(buf.status.abs().sum()) == 0
    return buf.U.view(H, T, 128)[:, 0].float().cpu().numpy().astype(np.float64)


def _neighbours(x, dtype):
    """The largest 16-bit value <= x and the smallest >= x (x: float64 of fp32 values)."""
    t16 = torch.tensor(x, dtype=torch.float32).to(NEIGHBOURS[dtype])
    r = t16.double().numpy()
    bits = t16.view(torch.int16).numpy().astype(np.int32)
    # one step toward +inf / -inf in the sign-magnitude encoding
    up = np.where(r >= 0, bits + 1, bits - 1)
    dn = np.where(r > 0, bits - 1, bits + 1)
    step = lambda b: torch.tensor(b.astype(np.int16)).view(NEIGHBOURS[dtype]).double().numpy()
    lo = np.where(r <= x, r, step(dn))
    hi = np.where(r >= x, r, step(up))
    return lo, hi


@pytest.mark.parametrize('dtype', ['bf16', 'f16'])
def test_stochastic_rounding_is_unbiased(dtype):
    # the appended key column stores k itself, so the value before rounding is known
    # exactly: the fp32 key
    rng = np.random.default_rng(5)
    k = rng.standard_normal(128)
    k = (k / np.linalg.norm(k)).astype(np.float32).astype(np.float64)
    H = 1024
    rn = _append_copies(dtype, 'nearest', 1, k)[0]
    sr = _append_copies(dtype, 'stochastic', H, k)
    near = torch.tensor(k, dtype=torch.float32).to(NEIGHBOURS[dtype]).double().numpy()
    assert np.array_equal(rn, near)                                       # nearest is nearest even
    lo, hi = _neighbours(k, dtype)
    assert np.all((lo <= k) & (k <= hi))
    assert np.all((sr == lo) | (sr == hi))                                # only the two neighbours
    moving = hi > lo
    assert moving.sum() > 100
    p = (sr == hi).mean(axis=0)[moving]                                   # fraction rounded up
    p_true = ((k - lo) / np.where(moving, hi - lo, 1.0))[moving]
    sd = np.sqrt(np.maximum(p_true * (1 - p_true), 1.0 / H) / H)
    z = (p - p_true) / sd
    assert np.max(np.abs(z)) < 6.0
    assert abs(np.mean(z)) < 0.3 and 0.6 < np.std(z) < 1.3               # mean k, binomial spread


@pytest.mark.parametrize('dtype', ['bf16', 'f16'])
def test_stochastic_rounding_is_reproducible(dtype):
    H, T, s = 24, 8, 8
    ranks = np.full(H, 16, np.int32)
    states, vbar = random_states(61, H, 128, 128, ranks, s, T, 'gdn', dtype)
    outs = []
    for seed in (11, 11, 12):
        buf = make_buffers('gdn', dtype, H, 128, 128, T, vbar, ranks, rounding='stochastic', sr_seed=seed)
        upload(buf, states, s)
        nb = R.seed_recompress_workspace_bytes(buf.st, H)
        ws = torch.empty(nb, device='cuda', dtype=torch.uint8)
        R.seed_recompress_ws(buf.st, None, None, ws, nb)
        torch.cuda.synchronize()
        outs.append((buf.U.clone(), buf.W.clone()))
        S = gpu_dense(buf)
        for h in range(H):
            ref, _ = oracle.recompress(states[h], int(ranks[h]))
            assert rel_err(S[h], oracle.materialize(ref)) < TOL[dtype], h
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert not torch.equal(outs[0][0], outs[2][0]) and not torch.equal(outs[0][1], outs[2][1])


def test_drift_by_storage_format(record_property):
    # a batched Gated DeltaNet trajectory (the 2,048-head workload's distributions,
    # 4 requests x 32 heads), 256 steps with a recompression every 16, in each storage
    # format; drift = relative Frobenius error of the reconstructed state against the
    # float64 oracle (no storage rounding), worst over sampled heads and steps
    from test_gpu_pipeline import gpu_head_states, oracle_head
    base = synth.GDN_BATCHED.with_(n_req=4)
    steps = base.steps
    heads = [0, 37, 77, 127]
    record = [16, 64, 128, 192, 255]
    ref = {}
    for h in heads:
        traj, _, _ = oracle_head(base, h, steps, record)
        ref[h] = traj
    drift = {}
    for dtype in ('bf16', 'f16'):
        for rounding in ('nearest', 'stochastic'):
            w = base.with_(factor_dtype=dtype)
            run = DeviceRun(w, rounding=rounding, sr_seed=1000)
            S = run.prefill()
            run.compress(S)
            got = {}
            for t in range(1, steps + 1):
                run.gen_inputs(t - 1)
                run.decode()
                if t in record:
                    got[t] = gpu_head_states(run.state, heads).double().cpu().numpy()
                if t % w.T == 0:
                    run.recompress(run.trunc)
            torch.cuda.synchronize()
            assert int(run.state.status[:run.H].abs().sum()) == 0
            errs = {t: max(rel_err(got[t][i], ref[h].states[t]) for i, h in enumerate(heads)) for t in record}
            drift[f'{dtype}_{rounding}'] = errs
    for k, errs in drift.items():
        record_property('parity', dict(case=f'drift {k}', tol=TOL['bf16'], heads=len(heads), steps=steps,
                                       **{f'step{t}': float(e) for t, e in errs.items()}))
        print(k, {t: f'{e:.2e}' for t, e in errs.items()})
        assert max(errs.values()) < TOL['bf16'], (k, errs)
