"""W8A8 INT8 fused Mixture-of-Experts layer for GB300 (sm_103a).

The compute runs in the CUDA library ``libwq.so`` (built from ``csrc/``)
behind the C ABI declared in ``include/wq.h``; ``binding`` marshals torch
tensors into those calls.  Importing this package does not load the library;
``binding.lib()`` does, and fails loudly if it is missing."""
