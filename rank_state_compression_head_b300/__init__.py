"""Python binding of libseed.so: sink + low-rank recurrent-state decode on B300.

Argument marshalling only.  Every computation runs in the CUDA kernels of
``libseed.so`` (built in-tree by ``build.py``); there is no Python or CPU
implementation of any step, and importing this package fails loudly when the
library has not been built.

The functions below carry the names of the C-ABI (``include/seed.h``,
``include/seed_synth.h``).  Pointer arguments accept a ``torch.Tensor`` (its
device pointer is passed), an ``int`` address, or ``None`` (NULL).  Streams
accept a ``torch.cuda.Stream``, an ``int`` handle or ``None`` (the current
torch stream).  A non-zero status raises ``SeedError``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, 'libseed.so')

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f'{LIB_PATH} is missing: build the CUDA library first '
        '(python rank_state_compression_head_b300/build.py). There is no CPU fallback.')

_lib = ctypes.CDLL(LIB_PATH)

# enums (seed.h)
SEED_OK = 0
SEED_ERR_INVALID_ARG = 1
SEED_ERR_UNSUPPORTED_SHAPE = 2
SEED_ERR_CAPACITY = 3
SEED_ERR_ALIGNMENT = 4
SEED_ERR_CUDA = 5
SEED_ERR_NOT_CONVERGED = 6
SEED_ERR_NONFINITE = 7
SEED_ERR_TIMEOUT = 8
SEED_GDN, SEED_KDA, SEED_MAMBA2 = 0, 1, 2
SEED_F32, SEED_BF16, SEED_F16 = 0, 1, 2
SEED_ROUND_NEAREST, SEED_ROUND_STOCHASTIC = 0, 1
SEED_MAX_COLUMNS = 64
VARIANTS = {'gdn': SEED_GDN, 'kda': SEED_KDA, 'mamba2': SEED_MAMBA2}
DTYPES = {'f32': SEED_F32, 'bf16': SEED_BF16, 'f16': SEED_F16}
ROUNDINGS = {'nearest': SEED_ROUND_NEAREST, 'stochastic': SEED_ROUND_STOCHASTIC}

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_f32 = ctypes.c_float


class seed_state(ctypes.Structure):
    """Mirror of ``seed_state`` in seed.h (same field order and types)."""
    _fields_ = [
        ('variant', _i32), ('factor_dtype', _i32), ('n_heads', _i32), ('d_k', _i32), ('d_v', _i32),
        ('T', _i32), ('r', _i32), ('r_max', _i32), ('steps_since_compress', _i32), ('rounding', _i32),
        ('rank', _vp), ('col_offset', _vp), ('a', _vp), ('U', _vp), ('W', _vp), ('scale', _vp),
        ('vbar', _vp), ('vbar_index', _vp), ('status', _vp), ('sr_seed', ctypes.c_uint64),
        ('head_order', _vp), ('class_end', _i32 * 4),
    ]


class seed_synth_workload(ctypes.Structure):
    """Mirror of ``seed_synth_workload`` in seed_synth.h."""
    _fields_ = [
        ('variant', _i32), ('n_req', _i32), ('n_layers', _i32), ('n_head', _i32), ('d_k', _i32),
        ('d_v', _i32), ('seed', _u32), ('prefill_len', _i32), ('prefill_lo', _i32),
        ('prefill_hi', _i32), ('rank', _i32), ('n_rank_choices', _i32), ('rank_choices', _i32 * 4),
        ('sink_lo', _f32), ('sink_hi', _f32), ('noise_std', _f32), ('alpha_lo', _f32),
        ('alpha_hi', _f32), ('beta_lo', _f32), ('beta_hi', _f32), ('a_lo', _f32), ('a_hi', _f32),
        ('dt_mu', _f32), ('dt_var', _f32),
    ]


_sp = ctypes.POINTER(seed_state)
_wp = ctypes.POINTER(seed_synth_workload)
_PROTOS = {
    'seed_columns_per_head': (_i32, [_i32, _i32, _i32]),
    'seed_status_string': (ctypes.c_char_p, [ctypes.c_int]),
    'seed_compress_dense': (ctypes.c_int, [_vp, _sp, _vp, _vp]),
    'seed_decode_step': (ctypes.c_int, [_sp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    'seed_recompress': (ctypes.c_int, [_sp, _vp, _vp]),
    'seed_recompress_ex': (ctypes.c_int, [_sp, _vp, _vp, _vp]),
    'seed_recompress_workspace_bytes': (ctypes.c_int, [_sp, _i32, _vp]),
    'seed_recompress_ws': (ctypes.c_int, [_sp, _vp, _vp, _vp, _i64, _vp]),
    'seed_recompress_noalloc': (ctypes.c_int, [_sp, _vp, _vp, _vp]),
    'seed_materialize': (ctypes.c_int, [_sp, _vp, _vp]),
    'seed_dense_decode_step': (ctypes.c_int, [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _vp, _vp]),
    'seed_synth_raw': (ctypes.c_int, [_u32, _i32, _i32, _u32, _u32, _i32, _i32, _vp, _vp]),
    'seed_synth_constants': (ctypes.c_int, [_wp, _vp, _vp, _vp, _vp, _vp, _vp]),
    'seed_synth_step_inputs': (ctypes.c_int, [_wp, _i32, _i32, _i64, _i32, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _vp]),
    'seed_synth_dense_prefill': (ctypes.c_int, [_wp, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    'seed_synth_dense_prefill_chunked': (ctypes.c_int, [_wp, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
}
for _name, (_res, _args) in _PROTOS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED_SYMBOLS = tuple(_PROTOS)


class SeedError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f'{fn}: {status_string(status)} (status {status})')
        self.status = status


def status_string(status: int) -> str:
    return _lib.seed_status_string(int(status)).decode()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != SEED_OK:
        raise SeedError(fn, status)


# ----------------------------------------------------------------------------
# seed.h
# ----------------------------------------------------------------------------

def seed_columns_per_head(variant: int, r: int, T: int) -> int:
    return int(_lib.seed_columns_per_head(variant, r, T))


def seed_compress_dense(S, st: seed_state, trunc_err=None, stream=None) -> None:
    _check('seed_compress_dense',
           _lib.seed_compress_dense(_ptr(S), ctypes.byref(st), _ptr(trunc_err), _stream(stream)))


def seed_decode_step(st: seed_state, q, k, v, gate, beta, A, o, stream=None) -> None:
    _check('seed_decode_step',
           _lib.seed_decode_step(ctypes.byref(st), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta),
                                 _ptr(A), _ptr(o), _stream(stream)))


def seed_recompress(st: seed_state, trunc_err=None, stream=None) -> None:
    _check('seed_recompress', _lib.seed_recompress(ctypes.byref(st), _ptr(trunc_err), _stream(stream)))


def seed_recompress_ex(st: seed_state, trunc_err=None, sweeps=None, stream=None) -> None:
    _check('seed_recompress_ex', _lib.seed_recompress_ex(ctypes.byref(st), _ptr(trunc_err), _ptr(sweeps),
                                                         _stream(stream)))


def seed_recompress_workspace_bytes(st: seed_state, heads: int) -> int:
    out = ctypes.c_int64(0)
    _check('seed_recompress_workspace_bytes',
           _lib.seed_recompress_workspace_bytes(ctypes.byref(st), int(heads), ctypes.addressof(out)))
    return int(out.value)


def seed_recompress_ws(st: seed_state, trunc_err=None, sweeps=None, workspace=None, workspace_bytes: int = 0,
                       stream=None) -> None:
    _check('seed_recompress_ws',
           _lib.seed_recompress_ws(ctypes.byref(st), _ptr(trunc_err), _ptr(sweeps), _ptr(workspace),
                                   int(workspace_bytes), _stream(stream)))


def seed_recompress_noalloc(st: seed_state, trunc_err=None, sweeps=None, stream=None) -> None:
    _check('seed_recompress_noalloc',
           _lib.seed_recompress_noalloc(ctypes.byref(st), _ptr(trunc_err), _ptr(sweeps), _stream(stream)))


def seed_materialize(st: seed_state, S_out, stream=None) -> None:
    _check('seed_materialize', _lib.seed_materialize(ctypes.byref(st), _ptr(S_out), _stream(stream)))


def seed_dense_decode_step(variant: int, n_heads: int, d_k: int, d_v: int, S, q, k, v, gate, beta,
                           A, dir_index, o, stream=None) -> None:
    _check('seed_dense_decode_step',
           _lib.seed_dense_decode_step(variant, n_heads, d_k, d_v, _ptr(S), _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(gate), _ptr(beta), _ptr(A), _ptr(dir_index), _ptr(o),
                                       _stream(stream)))


# ----------------------------------------------------------------------------
# seed_synth.h
# ----------------------------------------------------------------------------

def seed_synth_raw(seed: int, phase: int, field: int, time: int, entity0: int, n_entities: int,
                   n_blocks: int, out, stream=None) -> None:
    _check('seed_synth_raw', _lib.seed_synth_raw(seed, phase, field, time, entity0, n_entities,
                                                 n_blocks, _ptr(out), _stream(stream)))


def seed_synth_constants(w: seed_synth_workload, vbar=None, sink_scale=None, A=None, rank=None,
                         prompt_len=None, stream=None) -> None:
    _check('seed_synth_constants',
           _lib.seed_synth_constants(ctypes.byref(w), _ptr(vbar), _ptr(sink_scale), _ptr(A), _ptr(rank),
                                     _ptr(prompt_len), _stream(stream)))


def seed_synth_step_inputs(w: seed_synth_workload, phase: int, time: int, head0: int, n_heads: int,
                           vbar, sink_scale, q, k, v, gate, beta, stream=None) -> None:
    _check('seed_synth_step_inputs',
           _lib.seed_synth_step_inputs(ctypes.byref(w), phase, time, head0, n_heads, _ptr(vbar),
                                       _ptr(sink_scale), _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                                       _ptr(beta), _stream(stream)))


def seed_synth_dense_prefill(w: seed_synth_workload, head0: int, n_heads: int, prompt_len, vbar,
                             sink_scale, A, S_out, stream=None) -> None:
    _check('seed_synth_dense_prefill',
           _lib.seed_synth_dense_prefill(ctypes.byref(w), head0, n_heads, _ptr(prompt_len), _ptr(vbar),
                                         _ptr(sink_scale), _ptr(A), _ptr(S_out), _stream(stream)))


def seed_synth_dense_prefill_chunked(w: seed_synth_workload, head0: int, n_heads: int, prompt_len, vbar,
                                     sink_scale, A, S_out, stream=None) -> None:
    _check('seed_synth_dense_prefill_chunked',
           _lib.seed_synth_dense_prefill_chunked(ctypes.byref(w), head0, n_heads, _ptr(prompt_len),
                                                 _ptr(vbar), _ptr(sink_scale), _ptr(A), _ptr(S_out),
                                                 _stream(stream)))


from .state import FactoredStateBuffers, synth_workload_struct  # noqa: E402,F401
