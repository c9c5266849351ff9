"""CPU oracle for the ReplaySSM decode-state path.

TEST INFRASTRUCTURE.  This package is the plain, slow, obviously-correct
reference that the CUDA kernels are checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product (``ssm_decode_state_gb300``) never does, and this
package imports nothing from the product.  It shares no code with the CUDA
path: no kernels, headers, helpers or constant tables.

Everything is float64 numpy, written in the order the method is described:
the oracle is the *stepwise* recurrence (the definition the replay form must
reproduce exactly up to rounding), not the replay form itself.

Pages cited (the three web pages the method is described on):

* [AT Pulse] "NVIDIA and Princeton's ReplaySSM stores a checkpoint and recent
  inputs instead of full SSM state to speed up hybrid-model decoding"
  (at-pulse.com story 2558);
* [Clarity] "NVIDIA and Princeton cache SSM inputs in place of state to speed
  hybrid-model decoding" (theclarity.today);
* [WittyWires] "ReplaySSM cuts memory traffic to speed up hybrid-model
  decoding" (wittywires.com forum).

Modules:

* ``mamba2`` -- stepwise Mamba-2 SSM decode recurrence, plus scoring of draft
  tokens and acceptance of a prefix (speculative decoding as plain stepwise
  updates).
* ``gdn``    -- stepwise gated delta rule (Gated DeltaNet decode).
* ``ring``   -- integer model of the per-sequence ring of input records:
  append, flush (fold), verify and rollback pointer moves.
* ``fp8``    -- FP8 E4M3 encoder/decoder written from the OCP 8-bit floating
  point format definition, and the per-row read-copy quantiser.

Parity pins (tests marked ``not gpu``) tie each module to closed forms,
special cases, library routines and brute force on tiny inputs.
"""
from . import fp8, gdn, mamba2, ring  # noqa: F401
