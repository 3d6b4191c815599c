"""skinny_gemm_gb300 -- W4A16 group-64 skinny GEMM for GB300 (sm_103a).

The public calls (``mm``, ``mm_id``, ``unpack``, ``dequant``) live in
``skinny_gemm_gb300.ops`` and go through the C-ABI library ``libw4a16.so``;
the seeded input generator is ``skinny_gemm_gb300.synth``.  Importing the
package loads nothing native: the CUDA library is opened on first use and a
missing or unbuildable library raises instead of falling back to anything.
"""
__all__ = ["ops", "synth"]
