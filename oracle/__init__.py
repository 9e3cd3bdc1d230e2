"""CPU oracle for descriptor-guided masked attention (TEST INFRASTRUCTURE ONLY).

Plain, slow, obviously-correct restatements of what the CompileMask hot path computes, written
from the method's description ("CompileMask: Bridging the Gap Between Expressiveness and
Efficiency in Attention Masking", sections 2.1, 3.2.2, 3.3.1, 3.3.2) and from the mask rules of
the five synthetic workloads.  Floating point is fp64.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library never calls it, and it shares no code with the CUDA path:
its only common dependency is the seeded input generator ``masked_flashattention_gb300.workloads``,
which holds no masking or attention arithmetic.

Modules
  masks      dense visibility predicates, canonical Interval Tables, Tile-State Bitmaps
  attention  fp64 softmax attention forward and backward over a dense boolean mask

Every function is pinned by a ``-m "not gpu"`` test to something other than itself (closed-form
counts, library routines, autograd, finite differences, the paper's worked example).
"""
