"""CPU oracle for the TurboQuant hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, fp64 NumPy
restatement of what the method computes, written from the source pages
(TurboQuant, arXiv:2504.19874, as explained by the pages "TurboQuant 详解",
"turboquant-first-principles-walkthrough", "TurboQuant 和 RotorQuant 的真相"
and "sub-byte-kv-cache-quantization-turboquant").  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product library never imports,
links or executes anything here, and nothing here imports the product.

Modules
-------
codebook   Lloyd-Max scalar quantizer over the post-rotation coordinate
           density (Beta form of f_X, or its Gaussian limit).
rotation   Haar rotation from the QR of a Gaussian matrix (sign-fixed),
           Hadamard matrices (Sylvester, Paley q=11) and the randomized
           Hadamard rotation.
quantizer  TurboQuant_MSE / TurboQuant_Prod encode with exhaustive
           nearest-centroid search, canonical bit packing, dequantization.
attention  Inner-product scores and decode attention by explicit
           dequantization (no pre-rotated query, no fused algebra).

Parity status: every function is pinned by a ``-m "not gpu"`` test against
values the pages print, closed forms or library routines, except the exact
numeric centroids of the d=128 Beta codebooks for b=3 and b=4, which no page
prints.  Those are pinned only by invariants (stationarity, symmetry, the
distortion table and the upper bound): parity unpinned for those exact values.
"""

from . import codebook, rotation, quantizer, attention  # noqa: F401
