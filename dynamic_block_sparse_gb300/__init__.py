"""GB300-native query-aware dynamic block-sparse decode attention over a paged bf16 KV cache.

The compute path is libdsa.so (hand-written sm_103a CUDA kernels behind a C ABI declared in
``include/dsa.h``); :mod:`.binding` marshals torch tensors into it, :mod:`.pipeline` strings the
calls into the decode steps of top-K, hierarchical (LServe), threshold (PSA) and speculate-and-
repair (PRR) sparse attention, and :mod:`.workloads` generates seeded synthetic inputs.
"""

__version__ = "0.1.0"
