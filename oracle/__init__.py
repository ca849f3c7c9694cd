"""CPU oracle for the W4A16 / NF4 dequantize-and-multiply path.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
the test suite, the smoke check and the bench's CPU-baseline leg may call it.
It shares no code with the CUDA path.

It is a plain, slow, obviously correct restatement of what the pages on 4-bit
weight-only quantization describe:

* ``numerics``  -- round-to-nearest-even to fp16 / bf16 (the storage dtypes).
* ``int4``      -- asymmetric round-to-nearest INT4 quantization, one fp16 scale
                   and one 4-bit zero point per group of 128 rows along K,
                   optional act-order row->group map, 8-nibbles-per-word
                   packing, and dequantization.
* ``nf4``       -- the 16-entry normal-float codebook, blockwise absmax
                   quantization and dequantization.
* ``product``   -- the fp64 reference product Y = X . W_hat and the
                   tolerance checks used by the parity tests.
* ``accounting``-- byte counts of the packed checkpoint tensors.
* ``awq``       -- the AWQ checkpoint layout (codes packed along N in AWQ's
                   column order) and its re-arrangement into this layout.

Floating point work is done in fp64 unless a step is defined in a narrower
type (the fp16 scale, the fp32 NF4 product).  Every function names the
passage it follows.

Pinning status (what each part is checked against, besides itself):
numerics, int4, product and accounting are pinned by the tests under
``tests/test_oracle_*.py``.  The NF4 codebook is pinned by its invariants and
an independent bisection of the normal CDF; exact equality of that codebook
with the table shipped by bitsandbytes is *parity unpinned*, because the pages
do not print the table; so is equality of the NF4 double-quantization second
level with bitsandbytes', and of the AWQ layout with files written by AWQ's
own tools (the pages describe neither).
"""

from . import accounting, awq, int4, nf4, numerics, product  # noqa: F401
