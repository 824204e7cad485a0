"""Device buffers of a factored state, and the workload-recipe struct.

PyTorch provides the device memory; the ``seed_state`` struct handed to the
C-ABI points into these tensors.  No arithmetic of the method happens here.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (SEED_BF16, SEED_F32, SEED_KDA, VARIANTS, DTYPES, ROUNDINGS, seed_state,
               seed_synth_workload)


def _p(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


class FactoredStateBuffers:
    """Sink + factor storage for ``n_heads`` heads, laid out as ``seed.h`` describes.

    Uniform rank ``r`` (``ranks is None``): columns of head h start at
    ``h * (r + growth*T)``.  Ragged ranks: ``ranks`` [n_heads] int32 and
    per-head column offsets (an exclusive prefix sum of ``rank + growth*T``).
    ``vbar`` is the [n_dir, d_v] table of unit sink directions and
    ``vbar_index`` (optional) the direction of each head.  With ragged ranks and
    ``class_order`` (the default), the heads are also listed by column class
    (capacity ``rank + growth*T`` in (16c, 16c + 16]) for the per-class launches
    that ``seed.h`` describes.
    """

    def __init__(self, variant: str, factor_dtype: str, n_heads: int, d_k: int, d_v: int, T: int,
                 vbar: torch.Tensor, r: int = 0, ranks: Optional[torch.Tensor] = None,
                 vbar_index: Optional[torch.Tensor] = None, device='cuda', rounding: str = 'nearest',
                 sr_seed: int = 0, class_order: bool = True):
        self.variant = variant
        self.factor_dtype = factor_dtype
        self.n_heads, self.d_k, self.d_v, self.T = n_heads, d_k, d_v, T
        self.growth = 2 if variant == 'kda' else 1
        tdt = {'bf16': torch.bfloat16, 'f16': torch.float16, 'f32': torch.float32}[factor_dtype]
        dev = torch.device(device)
        if ranks is None:
            self.r_max = r
            self.cap = r + self.growth * T
            self.ranks = None
            self.col_offset = None
            self.head_order, self.class_end = None, [0, 0, 0, 0]
            n_cols = n_heads * self.cap
        else:
            self.ranks = ranks.to(device=dev, dtype=torch.int32).contiguous()
            r_host = self.ranks.cpu().to(torch.int64)
            self.r_max = int(r_host.max()) if n_heads else 0
            caps = r_host + self.growth * T
            offs = torch.zeros(n_heads, dtype=torch.int64)
            if n_heads > 1:
                offs[1:] = torch.cumsum(caps, 0)[:-1]
            self.col_offset = offs.to(dev)
            self.cap = None
            n_cols = int(caps.sum())
            r = self.r_max
            self.head_order, self.class_end = None, [0, 0, 0, 0]
            if class_order and n_heads:
                cls = torch.where(caps <= 16, torch.zeros_like(caps), (caps - 1) // 16).clamp(max=3)
                self.head_order = torch.argsort(cls, stable=True).to(device=dev, dtype=torch.int32)
                self.class_end = torch.cumsum(torch.bincount(cls, minlength=4), 0).tolist()
        self.r = r
        self.n_cols = n_cols
        self.a = torch.zeros(n_heads, d_k, device=dev)
        self.U = torch.zeros(max(n_cols, 1), d_k, device=dev, dtype=tdt)
        self.W = torch.zeros(max(n_cols, 1), d_v, device=dev, dtype=tdt)
        if variant == 'kda':
            self.scale = torch.ones(max(n_heads, 1), d_k, device=dev)
        else:
            self.scale = torch.ones(max(n_cols, 1), device=dev)
        self.status = torch.zeros(max(n_heads, 1), dtype=torch.int32, device=dev)
        self.vbar = vbar.to(device=dev, dtype=torch.float32).contiguous()
        self.vbar_index = None if vbar_index is None else vbar_index.to(device=dev, dtype=torch.int32).contiguous()
        self.st = seed_state(
            variant=VARIANTS[variant], factor_dtype=DTYPES[factor_dtype], n_heads=n_heads, d_k=d_k,
            d_v=d_v, T=T, r=r, r_max=self.r_max, steps_since_compress=0, rounding=ROUNDINGS[rounding],
            rank=_p(self.ranks), col_offset=_p(self.col_offset), a=_p(self.a), U=_p(self.U),
            W=_p(self.W), scale=_p(self.scale), vbar=_p(self.vbar), vbar_index=_p(self.vbar_index),
            status=_p(self.status), sr_seed=sr_seed, head_order=_p(self.head_order))
        for c in range(4):
            self.st.class_end[c] = int(self.class_end[c])

    @property
    def steps_since_compress(self) -> int:
        return self.st.steps_since_compress

    def head_cols(self, h: int):
        """(first column, rank, current columns) of head h (host-side bookkeeping)."""
        growth_cols = self.growth * self.st.steps_since_compress
        if self.ranks is None:
            return h * self.cap, self.r, self.r + growth_cols
        r = int(self.ranks[h])
        return int(self.col_offset[h]), r, r + growth_cols


def synth_workload_struct(w) -> seed_synth_workload:
    """Fill the C recipe struct from a workload description (duck-typed)."""
    s = seed_synth_workload()
    s.variant = VARIANTS[w.variant]
    s.n_req, s.n_layers, s.n_head = w.n_req, w.n_layers, w.n_head
    s.d_k, s.d_v = w.d_k, w.d_v
    s.seed = w.seed
    s.prefill_len = w.prefill_len
    s.prefill_lo, s.prefill_hi = w.prefill_range
    s.rank = w.rank
    s.n_rank_choices = len(w.rank_choices)
    for i, c in enumerate(w.rank_choices):
        s.rank_choices[i] = c
    s.sink_lo, s.sink_hi = w.sink_scale
    s.noise_std = w.noise_std
    s.alpha_lo, s.alpha_hi = w.alpha_range
    s.beta_lo, s.beta_hi = w.beta_range
    s.a_lo, s.a_hi = w.a_range
    s.dt_mu, s.dt_var = w.dt_mu, w.dt_var
    return s
