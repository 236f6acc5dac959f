"""fp64 CPU oracle for the fused normalization + GEMM path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls,
links or executes this module.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

The oracle is the plain definition of every operation, written in float64
numpy.  It shares no code, constants or helpers with the CUDA library.  Its
inputs are the bf16 values the GPU sees, widened exactly to float64.

Sources (cited by page title and section):

* [FNF-ru]  "Free normalization fusion" (aixai.ru blog, a Russian summary of the
  PyTorch blog post "Towards Free Normalization").
* [FNF-es]  "PyTorch: normalización casi gratis fusionando kernels"
  (noticias.mechatronicstore.cl).
* [TFN]     "Towards Free Normalization: Fusing Normalization into GEMM and
  Attention Kernels – PyTorch" (news.8syncdev.com abstract).
* [ATB]     Ascend ATB RMSNorm-fusion article (gsyq.cn), sections 1.1 and 1.2,
  used only for the textbook LayerNorm / RMSNorm definitions.

Every function is pinned by the CPU tests in ``tests/test_oracle_pins.py``
(closed forms, hand-derived golden vectors, brute force and float64 library
routines).  No function here is "parity unpinned".
"""
from .fnorm_oracle import (  # noqa: F401
    gemm,
    rmsnorm,
    layernorm,
    lazy_prenorm_gemm,
    gemm_postnorm,
    prenorm_affine_gemm,
    gemm_add_postnorm,
    lazy_prenorm_gemm_backward,
    gemm_postnorm_backward,
    gemm_postnorm_backward_regrouped,
)
