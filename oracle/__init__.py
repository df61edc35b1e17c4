"""Oracle for the quantized linear-layer forward Y = X . W_hat^T -- TEST INFRASTRUCTURE ONLY.

Plain, slow, CPU-only numpy restatement of what the three pages define.  Only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import it; the product (``quantized_weight_linear_gb300``,
its C-ABI library and kernels) never does, and this package imports nothing
from the product.  The only code both sides share is the seeded input
generator ``qlin_synth``, which holds no quantization arithmetic.

Sources (page title, section):

* SpQR page -- "Makale Bülteni — SpQR", section "İddia ve Gerçeklik: SpQR":
  weights split into a dense low-bit matrix plus a sparse fp16 outlier matrix
  of about 1% of the entries; the dense part is 3-bit with groups of 16 and
  bi-level statistics; 3.36-4.75 bits per parameter on average; the kernel
  unpacks the dense codes while it applies the sparse matrix.
* GPTQ page -- "Makale Bülteni — GPTQ", intro and "İddia ve Gerçeklik: GPTQ":
  4-bit weights quantized in groups (blocks of 128 given as the example),
  round-to-nearest as the baseline quantizer, weight-only (activations stay
  16-bit).
* SmoothQuant page -- "Makale Bülteni — SmoothQuant", section "İddia ve
  Gerçeklik: SmoothQuant": Y = (X diag(s)^-1)(diag(s) W), per-token int8
  activations, per-channel int8 weights, migration strength alpha around
  0.8-0.85.

Where the pages leave a step open, the module docstrings state the reading
taken (the same readings are listed in the repository's design notes).

Modules
-------
``fp``           fp16 / bf16 rounding and bf16 ulp in numpy.
``rtn``          asymmetric round-to-nearest group quantizer Q_b.
``gptq_w4``      W4 g128 codes, canonical packing, dequantization.
``spqr``         outlier selection, bi-level 3-bit g16 quantizer, CSR, dequantization.
``smoothquant``  smoothing factors, per-channel int8 weights, per-token int8 activations,
                 exact integer accumulation and the scale epilogue.
``forward``      fp64 reference forward, the tolerance bound, bits per parameter.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, grid-exact idempotence, brute force on small tiles,
the pages' own figures in ``tests/golden/``).  Model-level quality
(perplexity) has no dataset here and is not computed.
"""
from . import fp, rtn, gptq_w4, spqr, smoothquant, forward  # noqa: F401
