"""libditstream: bounded-activation DiT block forward for GB300 (sm_103a).

The compute path is the C-ABI shared library ``libditstream.so`` built from
``csrc/`` (hand-written CUDA for sm_103a); ``ditstream`` is its thin ctypes
binding and ``synth`` draws the seeded synthetic inputs.  Importing this
package loads nothing; ``ditstream.load()`` opens the library and raises if
it is missing (there is no CPU fallback).
"""

__all__ = ["synth", "ditstream"]
