"""fp64 CPU oracle for the OSCAR mixed-precision INT2 KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the C-ABI library, its
kernels or its Python binding) imports, links or executes this package; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg do.
It shares no code with the CUDA path: its inputs come from the seeded
generators in ``int2_rotated_kv_gb300.synth`` (which hold none of the method's
arithmetic) and from hand-written fixtures under ``tests/golden``.

Sources.  The method is defined by two web pages about arXiv 2605.17757:
  [Summary]  "Technical Summary: OSCAR - Offline Spectral Covariance-Aware
             Rotation for 2-bit KV Cache Quantization" (gist.science), cited by
             section, e.g. [Summary 2.2A.3] = section 2.2, phase A, step 3.
  [Abstract] "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
             Cache Quantization" (mlsanity.com index page), its arXiv abstract.
Where the pages are silent the modules state the reading they take.

Modules
  rotation   covariances C_Q, C_S; eigenbasis; normalised Hadamard; bit-reversal
             permutation; composite rotation R = U H P_br; clipping threshold.
  quant      rotate + clip + asymmetric INT2 group quantisation; dequantisation;
             the near-boundary flags used to compare against a kernel whose
             rotated value carries fp32 rounding error.
  layout     the library's page formats (where each code, scale, zero and bf16
             value of a page lives), written as index formulas.
  cache      expected page-pool contents for prefill and decode-append.
  attention  softmax attention over the mixed BF16 / INT2 cache, by the plain
             definition (reconstruct keys and values, then attend).

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
closed forms, textbook cases, library routines or brute force, except the
end-to-end fidelity numbers (OSCAR vs Hadamard-only vs unrotated), which the
pages print no numbers for: parity unpinned for ``attention.fidelity_report``.
"""
from . import attention, cache, layout, quant, rotation  # noqa: F401
