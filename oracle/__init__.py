"""CPU oracle for the routed-attention DiT block (test infrastructure only).

This package is the slow, plain reference that the CUDA path is checked
against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the product library never calls it and has no
CPU fallback.  It shares no code with the CUDA path: the only common module is
``synthetic`` (seeded input draws).

Arithmetic is float64 throughout, except where the method itself fixes a
precision: the bf16 "mids" that the pages declare (modulated-norm output,
projection outputs, head layout, attention output, residual stream) are
rounded to bf16 exactly where the method stores bf16, and the top-k decision
is taken on fp32 scores, the precision the FastH3 pages fix for routing.

``h3ref.c`` (loaded by ``cref.py``) restates the block once more in plain C
loops, written apart from the numpy code; the tests require the two to agree.

Every public function is pinned by tests in ``tests/test_oracle_pins.py``;
the pin table in the header of ``h3block.py`` names them.  The pages print no
worked example of a whole block or denoiser step (no weights or fixtures), so
the composed block and denoiser are pinned through closed-form special cases
of each of their stages, not by value on general inputs.
"""
from .h3block import *  # noqa: F401,F403
