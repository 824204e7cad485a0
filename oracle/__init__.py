"""CPU oracle for sink + low-rank recurrent-state decode.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA library and does not import it.

Everything here is plain float64 numpy, one head at a time, written from
"Shallow Encoding Emits Deep Memories" (SEED):

* the dense recurrences of Gated DeltaNet, Kimi Delta Attention and Mamba-2
  with the read-out of the updated state;
* the state sink split (Lemma 1) used to compress a dense state;
* the exact factored update (Lemma 2) for all three recurrences;
* periodic recompression to rank r (QR of both factors, SVD of the core,
  truncation) and the reconstruction of the dense state;
* the state-bytes model of the paper's Table 2 and the open-loop error bound
  of Corollary 4.

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (closed forms, constructed answers, brute force, the pages'
printed numbers).  See ``tests/test_oracle_*.py``.
"""
from .seed_oracle import *  # noqa: F401,F403
