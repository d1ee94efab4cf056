"""CPU oracle for the fused attention forward pass -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 restatements of what the pages define. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
or execute anything in this package; the library under
``online_softmax_fwd_gb300/`` never does, and this package never imports it.

Modules
  attention      one-shot softmax(Q K^T s) V and LSE (the definition), plus the
                 blockwise online recurrence used only to check the definition
                 against the identities the pages state, and the exact merge of
                 (O, LSE) results over disjoint key sets.
  exp2_model     the accuracy statistics of a software exp2 (the columns the
                 page prints) and a bf16 rounding from the value itself.
  cmodel         ctypes loader for ``exp2_model.c``: the software exp2 (range
                 reduction + degree-3 Horner) in scalar C with a fused
                 multiply-add, the one model of it, for bit-exact comparison.
  rescale_stats  the lagging-max (tau) rescale simulator and its statistics.
  mxfp8          the E4M3 / E8M0 32x32 block quantiser and its dequantisation.
  backward       the gradient of the forward (dQ, dK, dV) with P rebuilt from
                 the LSE: the five products of the backward pass, in float64
                 and with MXFP8 inputs (32 x 32 blocks for Q, K, V, dO, dS).

Parity pins (tests/test_oracle_*.py, marked "not gpu") tie every function here
to something other than itself: brute force, closed forms, and the numbers the
pages print. Degree-4 and degree-5 software exp2 are not built: their
coefficients are not printed, so they would be parity unpinned.
"""
