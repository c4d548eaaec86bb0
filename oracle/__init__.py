"""CPU oracle for layer-streamed NF4-LoRA (plain, slow, float64 numpy).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import or run anything in this package.  The product (the CUDA library
and its Python binding) never imports it, and it never imports the product.  The two share
no code, headers, tables or constants; only the seeded input generators in ``synth`` serve
both.

Modules:

* ``oracle.nf4``   -- NF4 codebook, blockwise quantisation with double-quantised absmax,
  packed byte layout, dequantisation.
* ``oracle.lora``  -- the frozen-base linear with its LoRA branch, forward and backward.
* ``oracle.stack`` -- the synthetic decoder layer, the 32-layer stack, its loss and the
  hand-derived backward.

Parity status: every function is pinned by the ``-m "not gpu"`` tests except the absolute
values of the NF4 codebook beyond what its construction fixes (see ``oracle.nf4``).
"""
