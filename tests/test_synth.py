"""The seeded input generator: Philox4x32-10 known answers and workload distributions."""
import numpy as np
import pytest

import synth


# Known-answer vectors published with the Random123 library (kat_vectors,
# philox4x32 with 10 rounds): counter words, key words, expected output.
PHILOX_KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff, 0xffffffff, 0xffffffff, 0xffffffff), (0xffffffff, 0xffffffff),
     (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
]


@pytest.mark.parametrize('ctr,key,expect', PHILOX_KAT)
def test_philox_known_answers(ctr, key, expect):
    out = synth.philox4x32_10(*ctr, *key)
    assert tuple(int(x) for x in out) == expect


def test_uniforms_open_interval_and_exact_in_fp32():
    x = np.array([0, 511, 512, 0xFFFFFFFF], dtype=np.uint32)
    u = synth.uniform_from_word(x)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert u[0] == 2 ** -24 and u[-1] == 1 - 2 ** -24


def test_normal_moments():
    z = synth.normals(7, synth.PHASE_DECODE, synth.FIELD_V, np.arange(2000), 3, 128)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1) < 0.01
    assert abs(np.mean(z ** 4) - 3) < 0.05


@pytest.mark.parametrize('name', list(synth.WORKLOADS))
def test_workload_inputs_shapes_and_ranges(name):
    w = synth.WORKLOADS[name]
    heads = np.array([0, 1, w.n_heads - 1])
    d = synth.decode_inputs(w, 3, heads)
    if w.variant == 'mamba2':
        assert d['C'].shape == (3, w.d_k) and d['x'].shape == (3, w.d_v)
        assert np.all(d['dt'] > 0)
        A = synth.mamba2_A(w)
        assert np.all((A <= -1) & (A >= -16))
    else:
        assert np.allclose(np.linalg.norm(d['q'], axis=1), 1, atol=1e-6)
        assert np.allclose(np.linalg.norm(d['k'], axis=1), 1, atol=1e-6)
        lo, hi = w.alpha_range
        assert np.all((d['alpha'] >= lo) & (d['alpha'] <= hi))
        lo, hi = w.beta_range
        assert np.all((d['beta'] >= lo) & (d['beta'] <= hi))
    vb = synth.sink_directions(w)
    assert vb.shape == (w.n_dir, w.d_v)
    assert np.allclose(np.linalg.norm(vb, axis=1), 1, atol=1e-6)


def test_ragged_ranks_and_prompt_lengths():
    w = synth.GDN_SERVING
    r = synth.head_ranks(w, np.arange(30000))
    assert set(np.unique(r)) == {16, 32, 48}
    assert all(abs(np.mean(r == c) - 1 / 3) < 0.02 for c in (16, 32, 48))
    L = synth.prompt_lengths(w)
    assert L.shape == (512,) and L.min() >= 512 and L.max() <= 8192
    assert synth.head_request(w, w.n_heads - 1) == 511 and synth.head_dir(w, 1152) == 0


def test_value_sink_component():
    # v = s vbar + noise: the projection on vbar averages to the sink scale
    w = synth.GDN_TINY
    d = synth.token_inputs(w, synth.PHASE_DECODE, np.arange(400)[:, None], np.arange(4)[None, :])
    vb = synth.sink_directions(w)
    proj = np.einsum('thd,hd->th', d['v'], vb)
    assert np.allclose(proj.mean(axis=0), 3.0, atol=0.1)
