"""CPU oracle for fine-grained-scaled FP8 (e4m3) GEMM.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously-correct
statement of what the GPU path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with ``fp8_fine_grained_e4m3_gb300`` (the CUDA path) and
never imports it; the product path never imports this package.

Pages it follows (no page prints a title, so each is named by its address):

* "news.rkmt.cn/news/5092" -- a DeepGEMM teardown (sections 1-6);
* "lpnh.cn/news/2822121" -- a DeepGEMM teardown (sections 1.1-6.3);
* "blog.hotdry.top: DeepGEMM FP8 GEMM fine-grained scaling kernels"
  (unnumbered sections, cited by their headings);
* "bhfrc.com/news/60211" -- a DeepGEMM user report (sections 1.1-7).

Modules:

* :mod:`oracle.e4m3`  -- the OCP E4M3 ("fn") code: decode table and
  round-to-nearest-even, saturating encoder.
* :mod:`oracle.e5m2`  -- the E5M2 code (IEEE-style infinities and NaNs),
  same two pieces.
* :mod:`oracle.quant` -- 1x128 (activations) and 128x128 (weights)
  quantisers, FP32 semantics.
* :mod:`oracle.gemm`  -- the block-scaled GEMM in FP64: dense, grouped
  contiguous, grouped masked, and a sampled-element form.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
library routines or brute force; nothing here is "parity unpinned".
"""

from . import e4m3, e5m2, quant, gemm  # noqa: F401
