"""Grammar-constrained logit masking and fused sampling for GB300 (sm_103a).

The compute path is the CUDA library ``liblp.so`` (sources in ``csrc/``, C-ABI in
``include/lp.h``); ``ops`` is a thin PyTorch-facing binding over it.  Importing
this package does not load the library; the first op call does, and fails loudly
if it has not been built.
"""

__all__ = ["ops", "synthetic"]
