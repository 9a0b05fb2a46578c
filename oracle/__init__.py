"""Plain CPU oracle for the fused GEMM epilogue hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the C-ABI library
and its Python binding) may import, call, link or execute anything in this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
and ``--impl reference`` legs of ``bench.py`` use it.

What it computes is the plain definition of the operation the QuACK pages
implement for Hopper (quack-kernels 0.2.0, ``quack/gemm_act_sm90.py``
``GemmActSm90.epi_visit_acc_subtile`` and ``quack/dense_gemm_sm90.py``
``GemmSm90.epi_visit_acc_subtile``)::

    D[m, n, l]       = rnd_D( alpha * sum_k A[m, k, l] * B[n, k, l] + beta * C[m, n, l] )
    PostAct[m, n, l] = rnd_P( act( alpha * sum_k ... + beta * C ) )

in float64 from the already-quantised input codes, with the activation
evaluated on the UNROUNDED value and each output rounded once,
round-to-nearest-even, to its storage format.  The varlen-M form walks
groups ``g`` whose rows are ``[cu_seqlens_m[g], cu_seqlens_m[g+1])`` against
``B[:, :, g]``; the gather form replaces row ``r`` of A by
``A_src[a_idx[r]]``.

Modules:
  formats     -- exact decoders and RNE encoders of bf16 / fp16 / fp32 /
                 float8_e4m3fn / float8_e5m2, written from the format
                 definitions.
  activations -- relu, gelu (tanh form), silu in float64.
  gemm        -- the GEMM + epilogue, varlen-M and gather-A definitions and the
                 per-element error bound used by the parity tests.
  fastdivmod  -- FastDivmod exactly as ``quack/fast_math.py`` builds it, in
                 Python integers.
  tiles       -- the set of output tiles a schedule must cover exactly once.

Every function is pinned by ``tests/test_oracle_pins.py`` against values fixed
by mathematics or by independent libraries.  No function here is
"parity unpinned".
"""

from . import formats, activations, gemm, fastdivmod, tiles  # noqa: F401
