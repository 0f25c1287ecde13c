"""CPU oracle for the trellis-coded MoE layer (TEST INFRASTRUCTURE ONLY).

This package is the plain, slow, float64 statement of what the layer
computes. It exists to check the CUDA path; it is not part of it. Only the
test suite, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg
and its ``--impl reference`` arm) may import or run it. The product path never
calls into this package and shares no code with it: the only code the two
sides have in common is the seeded input generator
``trellis_quantized_moe_route_gb300.synth``, which holds none of the layer's
arithmetic.

Sources (four pull-request pages; cited by title and section throughout):
  * b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms"
    (Summary, Hot path, review of trellis_w4a8.py);
  * b12x PR #433 "Share trellis preparation across native and EXL3 containers"
    (conversation, review of route_pack.py, Behavior);
  * sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused W4A16 API"
    (review of intrinsics.py, kernel.py, prepare.py, route_pack.py);
  * flashinfer PR #69 "b12x fused MoE: TrellisMX (procedural NPK) source
    format with an in-tree P8 runtime" (Description; Evidence, precision notes).

Modules:
  trellis   - bitstream, 16-bit tail-biting states, MCG codebook, tile decode
  hadamard  - Sylvester Hadamard matrices and blockwise rotation
  mxfp8     - E4M3 rounding and the UE8M0 (E8M0) block exponent
  route     - top-k softmax router and the stable route map
  layer     - the whole layer (W4A16 and W4A8)
  linear    - the dense trellis linear layer (one matrix, no routing; W4A16)

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, hand-computed values, invariants or brute force. One
point stays unpinned against any outside implementation: the pages print no
decoded codebook sample, so the way the three codebook constants combine
(mask then XOR) is a reading; see the ``trellis`` module docstring.
"""
