"""Per-class launches through the state's class order (needs a GPU).

seed.h: with head_order, the decode and the 16-bit recompression launch once per
column class, each launch sized for its class; the results must be those of the
single launch, head for head and bit for bit.  A head listed in a class too
small for it is reported (status 1) and left untouched.
"""
import numpy as np
import pytest
import torch

import rank_state_compression_head_b300 as R
from _gpu import make_buffers, random_states, upload

pytestmark = pytest.mark.gpu

D_V = {'gdn': 128, 'kda': 128, 'mamba2': 64}


def _ranks(variant, H, T):
    growth = 2 if variant == 'kda' else 1
    top = 64 - growth * T
    base = [1, 7, top, 16, 31, 5, top - 1, 24, 0, 12, 40 if top >= 40 else top]
    return np.array([base[h % len(base)] for h in range(H)], dtype=np.int32)


def _inputs(variant, H, T, seed):
    g = torch.Generator().manual_seed(seed)
    steps = []
    for _ in range(T):
        q = torch.randn(H, 128, generator=g)
        k = torch.randn(H, 128, generator=g)
        q, k = q / q.norm(dim=1, keepdim=True), k / k.norm(dim=1, keepdim=True)
        v = torch.randn(H, D_V[variant], generator=g)
        if variant == 'kda':
            gate = 0.8 + 0.19 * torch.rand(H, 128, generator=g)
        elif variant == 'mamba2':
            gate = 0.05 + 0.3 * torch.rand(H, generator=g)  # dt
        else:
            gate = 0.85 + 0.14 * torch.rand(H, generator=g)
        beta = 0.05 + 0.9 * torch.rand(H, generator=g)
        steps.append([t.cuda() for t in (q, k, v, gate, beta)])
    A = (-1.0 - 15.0 * torch.rand(H, generator=g)).cuda()
    return steps, A


def _run(buf, steps, A, H, variant):
    outs = []
    o = torch.empty(H, D_V[variant], device='cuda')
    for q, k, v, gate, beta in steps:
        R.seed_decode_step(buf.st, q, k, v, gate, None if variant == 'mamba2' else beta,
                           A if variant == 'mamba2' else None, o)
        outs.append(o.clone())
    nbytes = R.seed_recompress_workspace_bytes(buf.st, 7)  # several chunks, a ragged last one
    ws = torch.empty(nbytes, device='cuda', dtype=torch.uint8)
    err = torch.zeros(H, device='cuda')
    R.seed_recompress_ws(buf.st, err, None, ws, nbytes)
    torch.cuda.synchronize()
    return outs, err


@pytest.mark.parametrize('variant,dtype,rounding', [('gdn', 'bf16', 'nearest'), ('gdn', 'bf16', 'stochastic'),
                                                    ('kda', 'f16', 'nearest'), ('mamba2', 'bf16', 'nearest')])
def test_class_order_gives_the_same_results(variant, dtype, rounding):
    H, T = 29, 8
    ranks = _ranks(variant, H, T)
    states, vbar = random_states(77, H, 128, D_V[variant], ranks, 0, T, variant, dtype)
    bufs = []
    for order in (True, False):
        b = make_buffers(variant, dtype, H, 128, D_V[variant], T, vbar, ranks, rounding=rounding, sr_seed=5,
                         class_order=order)
        upload(b, states, 0)
        bufs.append(b)
    assert bufs[0].head_order is not None and bufs[1].head_order is None
    assert len(set(np.searchsorted(bufs[0].class_end, np.arange(H), side='right'))) > 1  # several classes
    steps, A = _inputs(variant, H, T, 3)
    res = [_run(b, steps, A, H, variant) for b in bufs]
    for o1, o2 in zip(res[0][0], res[1][0]):
        assert torch.equal(o1, o2)
    assert torch.equal(res[0][1], res[1][1])
    for name in ('a', 'U', 'W', 'scale', 'status'):
        assert torch.equal(getattr(bufs[0], name), getattr(bufs[1], name)), name
    assert int(bufs[0].status.abs().sum()) == 0


def test_head_in_too_small_a_class_is_reported_and_untouched():
    variant, dtype, H, T = 'gdn', 'bf16', 12, 8
    ranks = np.array([8, 40, 16, 24, 8, 40, 16, 24, 8, 40, 16, 24], dtype=np.int32)
    states, vbar = random_states(78, H, 128, 128, ranks, 0, T, variant, dtype)
    good = make_buffers(variant, dtype, H, 128, 128, T, vbar, ranks)
    bad = make_buffers(variant, dtype, H, 128, 128, T, vbar, ranks)
    upload(good, states, 0)
    upload(bad, states, 0)
    # head 1 (capacity 48, class 2) listed with the class-1 heads (capacity at most 32)
    order = bad.head_order.cpu().numpy().tolist()
    ends = list(bad.class_end)
    order.remove(1)
    order.insert(ends[0], 1)
    ends[1] += 1
    bad.head_order.copy_(torch.tensor(order, dtype=torch.int32))
    for c in range(4):
        bad.st.class_end[c] = ends[c]
    steps, A = _inputs(variant, H, T, 4)
    U0 = bad.U.clone()
    _run(good, steps[:1], A, H, variant)
    _run(bad, steps[:1], A, H, variant)
    st = bad.status.cpu().numpy()
    assert st[1] == R.SEED_ERR_INVALID_ARG and (np.delete(st, 1) == 0).all()
    c0, _, _ = bad.head_cols(1)
    assert torch.equal(bad.U[c0:c0 + 48], U0[c0:c0 + 48])
    for h in range(H):
        if h == 1:
            continue
        c, r, _ = good.head_cols(h)
        assert torch.equal(good.U[c:c + r + T], bad.U[c:c + r + T]), h
        assert torch.equal(good.a[h], bad.a[h]), h


def test_misfiled_heads_in_a_persistent_launch():
    """More heads than one launch keeps resident: each CTA walks several heads and
    refills its stage from one to the next; the misfiled ones among them are reported
    and left untouched, and every other head comes out as in a correct order."""
    variant, dtype, H, T = 'gdn', 'bf16', 2600, 8
    ranks = np.where(np.arange(H) % 50 == 7, 40, 16).astype(np.int32)  # capacity 24 (class 1), 48 (class 2)
    states, vbar = random_states(79, H, 128, 128, ranks, 0, T, variant, dtype)
    good = make_buffers(variant, dtype, H, 128, 128, T, vbar, ranks)
    bad = make_buffers(variant, dtype, H, 128, 128, T, vbar, ranks)
    upload(good, states, 0)
    upload(bad, states, 0)
    order = bad.head_order.cpu().numpy().tolist()
    ends = list(bad.class_end)
    misfiled = [h for h in range(H) if ranks[h] == 40][::3]
    for h in misfiled:
        order.remove(h)
    span = ends[1] - ends[0]
    for i, h in enumerate(misfiled):  # spread through the class-1 positions
        order.insert(ends[0] + (i * span) // len(misfiled) + i, h)
    ends[1] += len(misfiled)
    bad.head_order.copy_(torch.tensor(order, dtype=torch.int32))
    for c in range(4):
        bad.st.class_end[c] = ends[c]
    steps, A = _inputs(variant, H, T, 5)
    U0, a0 = bad.U.clone(), bad.a.clone()
    outs = []
    for buf in (good, bad):
        o = torch.empty(2, H, 128, device='cuda')
        for t, (q, k, v, gate, beta) in enumerate(steps[:2]):
            R.seed_decode_step(buf.st, q, k, v, gate, beta, None, o[t])
        outs.append(o)
    torch.cuda.synchronize()
    st = bad.status.cpu().numpy()
    assert (st[misfiled] == R.SEED_ERR_INVALID_ARG).all()
    assert (np.delete(st, misfiled) == 0).all() and int(good.status.abs().sum()) == 0
    bad_set = set(misfiled)
    for h in range(H):
        c, r, _ = good.head_cols(h)
        if h in bad_set:
            assert torch.equal(bad.U[c:c + r + T], U0[c:c + r + T]) and torch.equal(bad.a[h], a0[h]), h
            continue
        assert torch.equal(outs[0][:, h], outs[1][:, h]), h
        assert torch.equal(good.U[c:c + r + T], bad.U[c:c + r + T]), h
        assert torch.equal(good.W[c:c + r + T], bad.W[c:c + r + T]), h
        assert torch.equal(good.a[h], bad.a[h]), h
