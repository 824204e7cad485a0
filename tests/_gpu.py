"""Helpers for the GPU parity tests: move oracle states in and out of device buffers.

Comparisons are made on reconstructed dense states and on outputs, never on
factors (the factors carry SVD sign and rotation freedom).
"""
import numpy as np
import torch

import oracle
import rank_state_compression_head_b300 as R

# Tolerances of the parity bar: relative Frobenius / L2 error of reconstructed
# states and outputs, fp32 factors and bf16 storage with fp32 accumulation.
TOL = {'f32': 1e-4, 'bf16': 1e-2, 'f16': 1e-2}


def stored(x, dtype: str) -> np.ndarray:
    """Value an array holds after storing it in the factor dtype (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, np.float64), dtype=torch.float64)
    if dtype == 'bf16':
        return t.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    if dtype == 'f16':
        return t.to(torch.float32).to(torch.float16).to(torch.float64).numpy()
    return t.to(torch.float32).to(torch.float64).numpy()


def random_states(seed, H, d_k, d_v, ranks, s, T, variant, dtype):
    """Random oracle states with m_h = rank_h + growth*s columns, already rounded to storage."""
    import synth
    growth = 2 if variant == 'kda' else 1
    m = np.asarray(ranks) + growth * s
    cap = int(np.max(ranks)) + growth * T
    raw = synth.random_factored_state(seed, H, d_k, d_v, m, cap, variant)
    states = []
    for h in range(H):
        st = oracle.FactoredState(a=stored(raw['a'][h], 'f32'), U=stored(raw['U'][h, :m[h]].T, dtype),
                                  W=stored(raw['W'][h, :m[h]].T, dtype), vbar=raw['vbar'][h])
        if variant == 'kda':
            st.D = stored(raw['D'][h], 'f32')
        else:
            st.scale = stored(raw['scale'][h, :m[h]], 'f32')
        states.append(st)
    return states, raw['vbar']


def make_buffers(variant, dtype, H, d_k, d_v, T, vbar, ranks, ragged=True, rounding='nearest', sr_seed=0,
                 class_order=True):
    vb = torch.tensor(np.asarray(vbar), dtype=torch.float32)
    kw = dict(rounding=rounding, sr_seed=sr_seed)
    if ragged:
        kw['class_order'] = class_order
        return R.FactoredStateBuffers(variant, dtype, H, d_k, d_v, T, vb,
                                      ranks=torch.tensor(np.asarray(ranks), dtype=torch.int32), **kw)
    return R.FactoredStateBuffers(variant, dtype, H, d_k, d_v, T, vb, r=int(ranks[0]), **kw)


def upload(buf, states, s):
    """Write oracle states into device buffers (values must already be storage-exact)."""
    buf.st.steps_since_compress = s
    tdt = buf.U.dtype
    for h, st in enumerate(states):
        c0, r, m = buf.head_cols(h)
        assert m == st.m, (m, st.m)
        buf.a[h] = torch.tensor(st.a, dtype=torch.float32)
        if m:
            buf.U[c0:c0 + m] = torch.tensor(st.U.T, dtype=torch.float32).to(tdt)
            buf.W[c0:c0 + m] = torch.tensor(st.W.T, dtype=torch.float32).to(tdt)
        if st.D is not None:
            buf.scale[h] = torch.tensor(st.D, dtype=torch.float32)
        else:
            buf.scale[c0:c0 + m] = torch.tensor(st.scale, dtype=torch.float32)
    torch.cuda.synchronize()


def gpu_dense(buf) -> np.ndarray:
    S = torch.empty(buf.n_heads, buf.d_k, buf.d_v, device='cuda')
    R.seed_materialize(buf.st, S)
    torch.cuda.synchronize()
    return S.double().cpu().numpy()


def rel_err(x, ref) -> float:
    return float(np.linalg.norm(np.asarray(x) - np.asarray(ref)) / np.linalg.norm(ref))


def normwise_out_err(o, o_ref, S_ref, q) -> float:
    """|o - o_ref| / (|S_ref|_2 |q|): the read-out error scaled by what the state can produce."""
    return float(np.linalg.norm(o - o_ref) / (np.linalg.norm(S_ref, 2) * np.linalg.norm(q)))


def to_dev(x):
    return torch.tensor(np.asarray(x), dtype=torch.float32, device='cuda').contiguous()
