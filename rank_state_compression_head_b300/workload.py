"""Drive one synthetic workload through the library on the GPU.

Only C-ABI calls: constants, dense prefill with in-kernel prompt tokens,
compression at the end of the prefill, then the decode loop (inputs of each
step generated on the device, fused read-out + update, recompression every T
steps).  PyTorch only allocates the buffers.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (SEED_MAMBA2, VARIANTS, seed_compress_dense, seed_decode_step, seed_dense_decode_step,
               seed_recompress_ex, seed_recompress_workspace_bytes, seed_recompress_ws, seed_synth_constants,
               seed_synth_dense_prefill, seed_synth_dense_prefill_chunked,
               seed_synth_step_inputs)
from .state import FactoredStateBuffers, synth_workload_struct

PHASE_DECODE = 2


# Heads per recompression group: enough to keep every SM busy, a few GB of workspace.
DEFAULT_WS_HEADS = 65536


class DeviceRun:
    """Buffers and calls for one workload ``w`` (a ``synth.Workload``-like object).

    ``ws_heads`` > 0 recompresses through the three-phase path with a workspace
    for that many heads per group; 0 uses the single-kernel recompression."""

    def __init__(self, w, device='cuda', steps_buffered: int = 1, ws_heads: int = DEFAULT_WS_HEADS,
                 rounding: str = 'nearest', sr_seed: int = 0):
        self.w = w
        self.dev = torch.device(device)
        self.wst = synth_workload_struct(w)
        H, dk, dv = w.n_heads, w.d_k, w.d_v
        self.H = H
        self.variant = VARIANTS[w.variant]
        n_dir = w.n_dir
        f32 = dict(device=self.dev, dtype=torch.float32)
        self.vbar = torch.empty(n_dir, dv, **f32)
        self.sink = torch.empty(n_dir, **f32)
        self.A = torch.empty(n_dir, **f32) if w.variant == 'mamba2' else None
        self.ranks = torch.empty(H, device=self.dev, dtype=torch.int32)
        self.plen = torch.empty(w.n_req, device=self.dev, dtype=torch.int32)
        seed_synth_constants(self.wst, self.vbar, self.sink, self.A, self.ranks, self.plen)
        self.vbar_index = (torch.arange(H, device=self.dev, dtype=torch.int32) % n_dir)
        ragged = bool(w.rank_choices)
        self.state = FactoredStateBuffers(
            w.variant, w.factor_dtype, H, dk, dv, w.T, self.vbar, r=w.rank if not ragged else 0,
            ranks=self.ranks if ragged else None, vbar_index=self.vbar_index, device=self.dev,
            rounding=rounding, sr_seed=sr_seed)
        # stochastic rounding: every call that stores factor elements gets the next
        # seed of a fixed sequence (fresh bits per call, reproducible per run)
        self.stochastic = rounding == 'stochastic'
        self._sr_next = sr_seed
        nb = max(1, steps_buffered)
        self.q = torch.empty(nb, H, dk, **f32)
        self.k = torch.empty(nb, H, dk, **f32)
        self.v = torch.empty(nb, H, dv, **f32)
        self.gate = torch.empty(nb, H, dk, **f32) if w.variant == 'kda' else torch.empty(nb, H, **f32)
        self.beta = torch.empty(nb, H, **f32)
        self.o = torch.empty(H, dv, **f32)
        self.trunc = torch.zeros(max(H, 1), **f32)
        self.nb = nb
        self.ws, self.ws_bytes = None, 0
        self.ws_heads = ws_heads
        if ws_heads > 0 and H > 0:
            self.ws_bytes = seed_recompress_workspace_bytes(self.state.st, min(H, ws_heads))
            self.ws = torch.empty(self.ws_bytes, device=self.dev, dtype=torch.uint8)

    # -- setup ------------------------------------------------------------------
    def prefill(self, head0: int = 0, n: Optional[int] = None, out: Optional[torch.Tensor] = None,
                chunked: bool = True):
        """Dense fp32 prefill of heads [head0, head0+n) into ``out`` (allocated if None).

        ``chunked`` selects the chunkwise kernel (a chunk of tokens per pass);
        otherwise the token-serial one.  Both give the recurrence's state.
        """
        n = self.H - head0 if n is None else n
        if out is None:
            out = torch.empty(n, self.w.d_k, self.w.d_v, device=self.dev, dtype=torch.float32)
        fn = seed_synth_dense_prefill_chunked if chunked else seed_synth_dense_prefill
        fn(self.wst, head0, n, self.plen, self.vbar, self.sink, self.A, out)
        return out

    def compress(self, S: torch.Tensor, trunc_err: Optional[torch.Tensor] = None):
        self._sr_advance()
        seed_compress_dense(S, self.state.st, trunc_err)

    # -- decode loop --------------------------------------------------------------
    def gen_inputs(self, step: int, slot: int = 0):
        seed_synth_step_inputs(self.wst, PHASE_DECODE, step, 0, self.H, self.vbar, self.sink,
                               self.q[slot], self.k[slot], self.v[slot], self.gate[slot],
                               self.beta[slot])

    def _sr_advance(self):
        if self.stochastic:
            self._sr_next += 1
            self.state.st.sr_seed = self._sr_next

    def decode(self, slot: int = 0, stream=None):
        self._sr_advance()
        seed_decode_step(self.state.st, self.q[slot], self.k[slot], self.v[slot], self.gate[slot],
                         self.beta[slot], self.A, self.o, stream)

    def recompress(self, trunc_err: Optional[torch.Tensor] = None, stream=None, sweeps=None):
        self._sr_advance()
        if self.ws is not None:
            seed_recompress_ws(self.state.st, trunc_err, sweeps, self.ws, self.ws_bytes, stream)
        else:
            seed_recompress_ex(self.state.st, trunc_err, sweeps, stream)

    def decode_launches(self) -> int:
        """Kernels one decode step launches: one per column class present when the state
        carries a class order (16-bit factors), else one (mirrors decode.cu)."""
        st = self.state
        if st.head_order is None or self.w.factor_dtype == 'f32':
            return 1
        ends = [0] + list(st.class_end)
        return sum(1 for c in range(4) if ends[c + 1] > ends[c])

    def recompress_launches(self) -> int:
        """Kernels one recompression after T steps launches (bookkeeping of the count
        a benchmark reports; mirrors the launcher in recompress_split.cu)."""
        if self.ws is None:
            return 1
        st = self.state
        m_max = st.r_max + st.growth * self.w.T
        groups = -(-self.H // min(self.H, self.ws_heads))
        if st.ranks is None or m_max <= 16:
            return 3 * groups
        classes = -(-m_max // 16)
        if self.w.factor_dtype == 'f32':
            return 3 * groups * classes
        if st.head_order is not None:  # three launches per class present in each chunk
            chunk, n, ends = min(self.H, self.ws_heads), 0, [0] + list(st.class_end)
            for p0 in range(0, self.H, chunk):
                p1 = min(self.H, p0 + chunk)
                n += 3 * sum(1 for c in range(4) if min(ends[c + 1], p1) > max(ends[c], p0))
            return n
        return groups * (1 + 3 * classes)  # a class-list pass, then three launches per class

    def step(self, t: int, slot: int = 0, stream=None) -> bool:
        """Decode step t (1-based) with inputs already in ``slot``; recompress when T divides t."""
        self.decode(slot, stream)
        if t % self.w.T == 0:
            self.recompress(self.trunc, stream)
            return True
        return False

    def dense_step(self, S: torch.Tensor, slot: int = 0, o: Optional[torch.Tensor] = None, stream=None):
        o = self.o if o is None else o
        seed_dense_decode_step(self.variant, self.H, self.w.d_k, self.w.d_v, S, self.q[slot],
                               self.k[slot], self.v[slot], self.gate[slot], self.beta[slot], self.A,
                               self.vbar_index, o, stream)
