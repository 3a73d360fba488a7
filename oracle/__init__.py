"""Oracle for query-aware dynamic block-sparse decode attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it.  It shares no code with the CUDA library:
it is a plain, slow, float64 CPU restatement of what each decode step computes, written from the
three source pages:

* "PSA: Progressive Sparse Attention — Algorithm and System Co-design for Efficient Attention in
  LLM Serving" (cited as *PSA*),
* "LServe: Efficient Long-sequence LLM Serving with Unified Sparse Attention" (cited as *LServe*),
* "Predict, Reuse, and Repair: Accelerating Dynamic Sparse Attention for Long-Context LLM
  Decoding" (cited as *PRR*).

Every function is pinned by a ``-m "not gpu"`` test against facts that do not come from the oracle
itself (a library softmax, brute force, closed forms, hand-derived sequences).  No function here
is "parity unpinned".
"""

from .dsa_oracle import *  # noqa: F401,F403
