"""GB300-native speculative verify and all-layer replay commit for Gated
DeltaNet (GDN) layers.

The compute path is the C-ABI library ``libgdn_spec.so`` (hand-written CUDA
for sm_103a).  ``spec_decode_recurrent_gb300.api`` is a thin ctypes binding
with the library's names; ``workloads`` draws the seeded synthetic inputs.
Importing this package loads nothing; the library is loaded on first use
and a missing library is an error, never a fallback.
"""

__all__ = ["api", "workloads"]
