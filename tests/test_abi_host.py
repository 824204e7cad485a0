"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import rank_state_compression_head_b300 as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000          # a 16-byte-aligned non-null address: never dereferenced on the host


def declared_functions():
    names = set()
    for hdr in ('seed.h', 'seed_synth.h'):
        with open(os.path.join(ROOT, 'include', hdr)) as f:
            text = f.read()
        text = re.sub(r'/\*.*?\*/', '', text, flags=re.S)
        for m in re.finditer(r'^\s*(?:const\s+)?(?:int|int32_t|char)\s*\*?\s*(seed_\w+)\s*\(', text, re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert {'seed_compress_dense', 'seed_decode_step', 'seed_recompress', 'seed_materialize',
            'seed_dense_decode_step', 'seed_status_string'} <= names
    lib = ctypes.CDLL(R.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names == set(R.EXPORTED_SYMBOLS)


def test_struct_layout_matches_header(tmp_path):
    # 10 int32 fields, 9 pointers, the 64-bit stochastic-rounding seed, the class
    # order pointer and its four class ends
    assert ctypes.sizeof(R.seed_state) == 10 * 4 + 9 * 8 + 8 + 8 + 4 * 4
    assert R.seed_state.a.offset == 56
    # the C compiler's view of seed.h agrees field by field with the ctypes mirror
    gcc = shutil.which('gcc')
    if gcc is None:
        pytest.skip('no C compiler')
    names = [f[0] for f in R.seed_state._fields_]
    src = tmp_path / 'layout.c'
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "seed.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(seed_state));\n' +
                   ''.join(f'  printf("%zu\\n", offsetof(seed_state, {n}));\n' for n in names) +
                   '  return 0;\n}\n')
    exe = tmp_path / 'layout'
    subprocess.run([gcc, '-I', os.path.join(ROOT, 'include'), str(src), '-o', str(exe)], check=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(R.seed_state)
    assert out[1:] == [getattr(R.seed_state, n).offset for n in names]


def test_status_strings():
    for code in range(9):
        assert R.status_string(code)
    assert 'capacity' in R.status_string(R.SEED_ERR_CAPACITY)
    assert R.status_string(99) == 'unknown status'


def test_columns_per_head():
    assert R.seed_columns_per_head(R.SEED_GDN, 32, 16) == 48
    assert R.seed_columns_per_head(R.SEED_KDA, 32, 16) == 64
    assert R.seed_columns_per_head(R.SEED_MAMBA2, 16, 16) == 32


def make_state(**kw):
    st = R.seed_state(variant=R.SEED_GDN, factor_dtype=R.SEED_BF16, n_heads=4, d_k=128, d_v=128, T=16,
                      r=32, r_max=32, steps_since_compress=0, rounding=0, rank=None, col_offset=None,
                      a=FAKE, U=FAKE, W=FAKE, scale=FAKE, vbar=FAKE, vbar_index=None, status=None)
    for k, v in kw.items():
        setattr(st, k, v)
    return st


def decode(st, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, gate=FAKE, beta=FAKE, A=None, o=FAKE)
    p.update(ptrs)
    return R._lib.seed_decode_step(ctypes.byref(st), p['q'], p['k'], p['v'], p['gate'], p['beta'],
                                   p['A'], p['o'], None)


@pytest.mark.parametrize('kw,code', [
    (dict(d_k=64), R.SEED_ERR_UNSUPPORTED_SHAPE),
    (dict(d_v=96), R.SEED_ERR_UNSUPPORTED_SHAPE),
    (dict(r=129, r_max=129), R.SEED_ERR_UNSUPPORTED_SHAPE),
    (dict(r=56, r_max=56), R.SEED_ERR_UNSUPPORTED_SHAPE),            # 56 + 16 > 64 columns
    (dict(variant=R.SEED_KDA, r=48, r_max=48), R.SEED_ERR_UNSUPPORTED_SHAPE),  # 48 + 32 > 64
    (dict(variant=7), R.SEED_ERR_INVALID_ARG),
    (dict(factor_dtype=3), R.SEED_ERR_INVALID_ARG),
    (dict(n_heads=-1), R.SEED_ERR_INVALID_ARG),
    (dict(T=0), R.SEED_ERR_INVALID_ARG),
    (dict(r=-1, r_max=-1), R.SEED_ERR_INVALID_ARG),
    (dict(a=None), R.SEED_ERR_INVALID_ARG),
    (dict(U=FAKE + 4), R.SEED_ERR_ALIGNMENT),
    (dict(scale=FAKE + 4), R.SEED_ERR_ALIGNMENT),
    (dict(steps_since_compress=16), R.SEED_ERR_CAPACITY),
])
def test_decode_rejects_on_host(kw, code):
    st = make_state(**kw)
    before = st.steps_since_compress
    assert decode(st) == code
    assert st.steps_since_compress == before


def test_decode_rejects_missing_inputs():
    st = make_state()
    assert decode(st, q=None) == R.SEED_ERR_INVALID_ARG
    assert decode(st, beta=None) == R.SEED_ERR_INVALID_ARG
    assert decode(st, o=FAKE + 8) == R.SEED_ERR_ALIGNMENT
    kda = make_state(variant=R.SEED_KDA, r=16, r_max=16)
    assert decode(kda, gate=FAKE + 4) == R.SEED_ERR_ALIGNMENT
    m2 = make_state(variant=R.SEED_MAMBA2, d_v=64, r=16, r_max=16)
    assert decode(m2, A=None, beta=None) == R.SEED_ERR_INVALID_ARG
    assert R._lib.seed_decode_step(None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None) == R.SEED_ERR_INVALID_ARG


@pytest.mark.parametrize('ends', [(1, 0, 2, 4), (0, 1, 2, 3), (0, 0, 0, 5), (-1, 0, 0, 4)])
def test_class_order_rejected_on_host(ends):
    # class ends must not decrease and must end at n_heads; checked before any launch
    st = make_state(rank=FAKE, r_max=32, head_order=FAKE)
    for c in range(4):
        st.class_end[c] = ends[c]
    before = st.steps_since_compress
    assert decode(st) == R.SEED_ERR_INVALID_ARG
    assert st.steps_since_compress == before
    f = R._lib.seed_recompress_ws
    st.steps_since_compress = 16
    assert f(ctypes.byref(st), None, None, FAKE, 1 << 30, None) == R.SEED_ERR_INVALID_ARG
    assert st.steps_since_compress == 16


def test_zero_heads_is_a_no_op_that_advances_the_counter():
    st = make_state(n_heads=0, a=None, U=None, W=None, scale=None, vbar=None)
    for s in range(16):
        assert decode(st, q=None, k=None, v=None, gate=None, beta=None, o=None) == R.SEED_OK
        assert st.steps_since_compress == s + 1
    assert decode(st) == R.SEED_ERR_CAPACITY
    assert R._lib.seed_recompress(ctypes.byref(st), None, None) == R.SEED_OK
    assert st.steps_since_compress == 0
    assert R._lib.seed_materialize(ctypes.byref(st), None, None) == R.SEED_OK
    assert R._lib.seed_compress_dense(None, ctypes.byref(st), None, None) == R.SEED_OK


def test_other_calls_reject_on_host():
    st = make_state()
    assert R._lib.seed_compress_dense(None, ctypes.byref(st), None, None) == R.SEED_ERR_INVALID_ARG
    assert R._lib.seed_compress_dense(FAKE + 4, ctypes.byref(st), None, None) == R.SEED_ERR_ALIGNMENT
    assert R._lib.seed_materialize(ctypes.byref(st), None, None) == R.SEED_ERR_INVALID_ARG
    st.steps_since_compress = 17
    assert R._lib.seed_recompress(ctypes.byref(st), None, None) == R.SEED_ERR_CAPACITY
    f = R._lib.seed_dense_decode_step
    assert f(0, 4, 64, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None) == R.SEED_ERR_UNSUPPORTED_SHAPE
    assert f(0, 4, 128, 128, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None) == R.SEED_ERR_INVALID_ARG
    assert f(2, 4, 128, 64, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, None) == R.SEED_ERR_INVALID_ARG
    assert f(0, 0, 128, 128, None, None, None, None, None, None, None, None, None, None) == R.SEED_OK


def test_synth_calls_reject_on_host():
    import synth
    w = R.synth_workload_struct(synth.GDN_BATCHED)
    bad = R.synth_workload_struct(synth.GDN_BATCHED.with_(d_k=64))
    assert R._lib.seed_synth_constants(ctypes.byref(bad), None, None, None, None, None, None) == R.SEED_ERR_UNSUPPORTED_SHAPE
    assert R._lib.seed_synth_step_inputs(ctypes.byref(w), 2, 0, 0, 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == R.SEED_ERR_INVALID_ARG
    assert R._lib.seed_synth_dense_prefill(ctypes.byref(w), 0, 0, None, None, None, None, None, None) == R.SEED_OK
    assert R._lib.seed_synth_raw(0, 0, 0, 0, 0, 4, 4, FAKE + 4, None) == R.SEED_ERR_ALIGNMENT


def _ws_floats(m, r, dk, dv, dtype='bf16'):
    # 16-bit factors (Cholesky of the value-side Gram matrix): M and R_b (rows of m4
    # floats), Y and eight words of class lists; 32-bit factors (QR of both factors):
    # W's reflectors, their tau, R_b^T, K, Y; each region on 16 bytes, the whole on
    # 256 bytes
    m4 = (m + 3) // 4 * 4
    mm4 = (m * m + 3) // 4 * 4
    if dtype == 'f32':
        n = m * dv + m4 + 2 * mm4 + r * m4
    else:
        n = 2 * m * m4 + r * m4 + 8
    n = (n + 63) // 64 * 64
    return max(n, 64)


def test_recompress_workspace_bytes():
    st = make_state()                                   # gdn, r = 32, T = 16, d_v = 128
    assert R.seed_recompress_workspace_bytes(st, 1) == 4 * _ws_floats(48, 32, 128, 128)
    assert R.seed_recompress_workspace_bytes(st, 1000) == 1000 * 4 * _ws_floats(48, 32, 128, 128)
    kda = make_state(variant=R.SEED_KDA, r=16, r_max=16, T=8)
    assert R.seed_recompress_workspace_bytes(kda, 3) == 3 * 4 * _ws_floats(32, 16, 128, 128)
    m2 = make_state(variant=R.SEED_MAMBA2, d_v=64, r=16, r_max=16)
    assert R.seed_recompress_workspace_bytes(m2, 2) == 2 * 4 * _ws_floats(32, 16, 128, 64)
    f32 = make_state(factor_dtype=R.SEED_F32)
    assert R.seed_recompress_workspace_bytes(f32, 5) == 5 * 4 * _ws_floats(48, 32, 128, 128, 'f32')
    out = ctypes.c_int64(0)
    f = R._lib.seed_recompress_workspace_bytes
    assert f(ctypes.byref(st), 0, ctypes.addressof(out)) == R.SEED_ERR_INVALID_ARG
    assert f(ctypes.byref(st), 4, None) == R.SEED_ERR_INVALID_ARG
    assert f(ctypes.byref(make_state(d_k=64)), 4, ctypes.addressof(out)) == R.SEED_ERR_UNSUPPORTED_SHAPE


def test_recompress_ws_rejects_on_host():
    f = R._lib.seed_recompress_ws
    st = make_state(steps_since_compress=16)
    one_head = 4 * _ws_floats(48, 32, 128, 128)
    assert f(ctypes.byref(st), None, None, None, one_head, None) == R.SEED_ERR_INVALID_ARG
    assert f(ctypes.byref(st), None, None, FAKE + 4, one_head, None) == R.SEED_ERR_ALIGNMENT
    assert f(ctypes.byref(st), None, None, FAKE, one_head - 4, None) == R.SEED_ERR_INVALID_ARG
    assert f(ctypes.byref(st), None, None, FAKE, -1, None) == R.SEED_ERR_INVALID_ARG
    st.steps_since_compress = 17
    assert f(ctypes.byref(st), None, None, FAKE, one_head, None) == R.SEED_ERR_CAPACITY
    assert st.steps_since_compress == 17
    empty = make_state(n_heads=0, a=None, U=None, W=None, scale=None, vbar=None, steps_since_compress=5)
    assert f(ctypes.byref(empty), None, None, None, 0, None) == R.SEED_OK
    assert empty.steps_since_compress == 0


def test_recompress_noalloc_rejects_oversize_before_cuda():
    f = R._lib.seed_recompress_noalloc
    per_head = _ws_floats(48, 32, 128, 128)
    limit = 16 << 20                                    # 64 MiB of fp32 scratch
    n_over = limit // per_head + 1
    st = make_state(n_heads=n_over, steps_since_compress=16)
    assert f(ctypes.byref(st), None, None, None) == R.SEED_ERR_UNSUPPORTED_SHAPE
    assert st.steps_since_compress == 16
    st.steps_since_compress = 17
    assert f(ctypes.byref(st), None, None, None) == R.SEED_ERR_CAPACITY
    empty = make_state(n_heads=0, a=None, U=None, W=None, scale=None, vbar=None, steps_since_compress=3)
    assert f(ctypes.byref(empty), None, None, None) == R.SEED_OK
    assert empty.steps_since_compress == 0
