"""seed_recompress_noalloc: the three-phase recompression on the library's own
fixed device scratch (needs a GPU).  Collected last, so that it runs both after
every other test in the session and alone.

It must give the same bits as seed_recompress_ws with a caller workspace, on
two recompressions in a row.
"""
import numpy as np
import pytest
import torch

import rank_state_compression_head_b300 as R
from _gpu import make_buffers, random_states, upload

pytestmark = pytest.mark.gpu


def _ranks(H, T):
    base = [32, 7, 31, 16, 1, 24, 0, 32 - 3]
    return np.array([base[h % len(base)] for h in range(H)], dtype=np.int32)


def _snapshot(buf, err, sweeps):
    torch.cuda.synchronize()
    return [x.clone() for x in (buf.U, buf.W, buf.scale, buf.a, buf.status, err, sweeps)]


@pytest.mark.parametrize('variant,dtype', [('gdn', 'bf16'), ('kda', 'bf16'), ('mamba2', 'f32')])
def test_noalloc_matches_workspace_call_twice(variant, dtype):
    H, T = 40, 16 if variant != 'kda' else 8
    d_v = 64 if variant == 'mamba2' else 128
    ranks = _ranks(H, T)
    one_ws, two_ws = None, None
    for call in range(2):
        s = T if call == 0 else T // 2
        states, vbar = random_states(71 + call, H, 128, d_v, ranks, s, T, variant, dtype)
        if one_ws is None:
            one = make_buffers(variant, dtype, H, 128, d_v, T, vbar, ranks)
            two = make_buffers(variant, dtype, H, 128, d_v, T, vbar, ranks)
            nbytes = R.seed_recompress_workspace_bytes(two.st, H)
            two_ws = torch.empty(nbytes, device='cuda', dtype=torch.uint8)
        upload(one, states, s)
        upload(two, states, s)
        e1, e2 = torch.zeros(H, device='cuda'), torch.zeros(H, device='cuda')
        w1 = torch.zeros(H, device='cuda', dtype=torch.int32)
        w2 = torch.zeros(H, device='cuda', dtype=torch.int32)
        R.seed_recompress_noalloc(one.st, e1, w1)
        R.seed_recompress_ws(two.st, e2, w2, two_ws, nbytes)
        assert one.st.steps_since_compress == 0
        for x, y in zip(_snapshot(one, e1, w1), _snapshot(two, e2, w2)):
            assert torch.equal(x, y)
        assert int(one.status.abs().sum()) == 0
        one_ws = True


def test_noalloc_rejects_oversize_without_launch():
    # enough heads at m = 48, r = 32 that their per-head workspace (the size that
    # seed_recompress_workspace_bytes reports at full capacity) no longer fits in
    # the 64 MiB scratch
    T = 16
    probe = make_buffers('gdn', 'bf16', 1, 128, 128, T, np.ones((1, 128)) / np.sqrt(128),
                         np.full(1, 32, dtype=np.int32), ragged=False)
    per_head = R.seed_recompress_workspace_bytes(probe.st, 1)
    H = (64 << 20) // per_head + 16
    ranks = np.full(H, 32, dtype=np.int32)
    vbar = np.ones((H, 128)) / np.sqrt(128)
    buf = make_buffers('gdn', 'bf16', H, 128, 128, T, vbar, ranks, ragged=False)
    buf.st.steps_since_compress = T
    with pytest.raises(R.SeedError) as e:
        R.seed_recompress_noalloc(buf.st)
    assert e.value.status == R.SEED_ERR_UNSUPPORTED_SHAPE
    assert buf.st.steps_since_compress == T


def test_noalloc_leaves_device_memory_unchanged():
    # The point of the call: nothing is allocated.  After one call (which loads the
    # kernels it launches), a second call changes neither the free device memory the
    # driver reports nor what the caching allocator holds.
    H, T = 40, 16
    ranks = _ranks(H, T)
    states, vbar = random_states(91, H, 128, 128, ranks, T, T, 'gdn', 'bf16')
    buf = make_buffers('gdn', 'bf16', H, 128, 128, T, vbar, ranks)
    err = torch.zeros(H, device='cuda')
    upload(buf, states, T)
    R.seed_recompress_noalloc(buf.st, err)
    upload(buf, states, T)
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    R.seed_recompress_noalloc(buf.st, err)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert int(buf.status.abs().sum()) == 0
