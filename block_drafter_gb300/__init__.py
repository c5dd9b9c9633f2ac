"""GB300 (sm_103a) block drafter: one DFlash-style parallel draft round with DSpine's
adjacent gated causal injection behind a small C ABI (``include/blockdrafter.h``).

Build the library with ``block_drafter_gb300.build.build()``; the binding in
``block_drafter_gb300.binding`` marshals torch tensors into the C calls.
"""
from .builder import LIBPATH, build  # noqa: F401
