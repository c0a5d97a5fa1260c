"""Reshard oracle: TEST INFRASTRUCTURE, not part of the product path.

A plain, slow, obviously correct CPU reference for what the reshard hot path computes. Only
the tests, the package entry's smoke check and the bench's CPU-baseline leg may import,
call, link or execute anything here. It shares no code with the CUDA path and neither side
imports the other; the only thing both use is the seeded input generator in ``synthetic``.

Two implementations that cross-check each other:
- ``oracle.golden`` (Python + numpy): the golden full-broadcast-then-slice semantics, the
  brute-force source-region enumeration and the one-element mapping used for sampled
  parity at full size.
- ``oracle.c`` (plain scalar C, built into ``liboracle.so`` and loaded by ``oracle.coracle``):
  the same semantics for the large workloads, streaming one tensor at a time.
- ``oracle.mxfp8`` (Python ints/fractions): the OCP MX v1.0 BF16 -> MXFP8 block rule.

Parity status of each function is stated in its module header.
"""
