"""CPU oracle for the NVFP4 MoE expert FFN.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The CUDA library never calls it, and this package imports nothing from
the CUDA library (``nvfp4_block_scaled_moe_gb300``): the two share no code.

Plain, slow, obviously-correct restatements of what the method computes, in the
order and notation of the source pages ("nvfp4-megamoe-kernel" notes):

* ``oracle.nvfp4`` -- FP8 E4M3 and FP4 E2M1 codecs, the per-16 block quantiser
  (scale = E4M3(amax/6), two-stage half-step E2M1 rounding), nibble packing and
  the swizzled scale-factor (SF) layout.
* ``oracle.moe``   -- top-k routing, the 128-padded expert permutation, the
  float64 block-scaled GEMM on dequantised operands, SwiGLU on the interleaved
  gate/up columns, and the routing-weighted combine.

Parity pins: every function is pinned in ``tests/test_oracle_*.py`` against
values the pages print (``tests/golden/``), closed forms, library routines
(PyTorch's float8_e4m3fn cast, numpy matmul) and brute force on tiny inputs.
The E2M1 half-step table entries hs=5 and hs=7 are not printed by the pages
(they print hs=10 and hs=11); they follow the ties-to-even reading stated in
``oracle.nvfp4.step_to_idx``, which the tests pin to PyTorch's independent
reference rounding to E2M1.
"""
