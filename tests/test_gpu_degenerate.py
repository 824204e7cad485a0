"""Recompression where the r-th and (r+1)-th singular values tie or nearly tie (needs a GPU).

With sigma_r = sigma_{r+1} several rank-r truncations are optimal, so the
truncated state is not unique and comparing it with the oracle's element by
element is ill-posed.  What is unique is the truncation error (Eckart-Young,
"Shallow Encoding Emits Deep Memories", picx.dev summary, Lemma 1 and its
truncation to rank R): sqrt of the sum of the discarded sigma^2.  So the test
checks (1) the reported truncation error against the oracle's, and (2) that the
GPU's own rank-r state is an optimal one: its distance to the state before the
recompression equals that error, to the parity tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_state_compression_head_b300 as R
from _gpu import TOL, gpu_dense, make_buffers, stored, upload

pytestmark = pytest.mark.gpu


def _tied_states(seed, H, r, m, variant, dtype, tie):
    """Heads with factor part X diag(sigma) Y^T, X and Y orthonormal, where
    sigma_{r-1} and sigma_r (0-based: the last kept and the first dropped) differ by
    the relative gap `tie` (0: an exact tie before storage rounding); for tie < 0
    three values straddle the boundary (r-2, r-1, r equal)."""
    rng = np.random.default_rng(seed)
    d_k = d_v = 128
    states, vbars = [], []
    for h in range(H):
        sig = 4.0 * 2.0 ** (-np.arange(m) / 6.0)
        c = 0.5 * (sig[r - 1] + sig[r])
        if tie < 0:
            sig[r - 2:r + 1] = c
        else:
            sig[r - 1], sig[r] = c * (1.0 + tie), c
        sig[r + 1:] = np.minimum(sig[r + 1:], 0.9 * c)
        X, _ = np.linalg.qr(rng.standard_normal((d_k, m)))
        Y, _ = np.linalg.qr(rng.standard_normal((d_v, m)))
        vbar = rng.standard_normal(d_v)
        vbar /= np.linalg.norm(vbar)
        st = oracle.FactoredState(a=stored(0.3 * rng.standard_normal(d_k), 'f32'),
                                  U=stored(X * sig[None, :], dtype), W=stored(Y, dtype), vbar=vbar)
        if variant == 'kda':
            st.D = np.ones(d_k)
        else:
            st.scale = np.ones(m)
        states.append(st)
        vbars.append(vbar)
    return states, np.array(vbars)


@pytest.mark.parametrize('variant,dtype', [('gdn', 'f32'), ('gdn', 'bf16'), ('gdn', 'f16'), ('kda', 'bf16')])
@pytest.mark.parametrize('tie', [0.0, 1e-6, 1e-3, -1.0], ids=['exact', 'near', 'close', 'triple'])
def test_recompress_at_a_singular_value_tie(variant, dtype, tie):
    H, T, r = 12, 8, 24
    growth = 2 if variant == 'kda' else 1
    m = r + growth * T
    states, vbar = _tied_states(7, H, r, m, variant, dtype, tie)
    ranks = np.full(H, r, dtype=np.int32)
    buf = make_buffers(variant, dtype, H, 128, 128, T, vbar, ranks)
    upload(buf, states, T)
    nbytes = R.seed_recompress_workspace_bytes(buf.st, H)
    ws = torch.empty(nbytes, device='cuda', dtype=torch.uint8)
    err = torch.zeros(H, device='cuda')
    R.seed_recompress_ws(buf.st, err, None, ws, nbytes)
    torch.cuda.synchronize()
    assert int(buf.status.abs().sum()) == 0
    S_gpu = gpu_dense(buf)
    err = err.double().cpu().numpy()
    tol = TOL[dtype]
    for h in range(H):
        S_before = oracle.materialize(states[h])
        _, e_ref = oracle.recompress(states[h], r)
        nrm = np.linalg.norm(S_before)
        # (1) the reported truncation error is the unique optimal one
        assert abs(err[h] - e_ref) <= tol * e_ref, (h, err[h], e_ref)
        # (2) the GPU's rank-r state is optimal: its distance to the state it replaced is
        # the truncation error, up to the parity tolerance (storage rounding of the new
        # factors included)
        dist = np.linalg.norm(S_gpu[h] - S_before)
        assert abs(dist - e_ref) <= tol * nrm, (h, dist, e_ref, nrm)
