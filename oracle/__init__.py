"""CPU oracle for topology-scheduled sparse attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  It shares no code with the CUDA library.
"""
from .oracle import (BF16, F16, attention, attention_backward, build, build_schedule, centroids, decode,  # noqa: F401
                     dense_causal_csr, fixed_segment_csr, max_nnz, pairwise_d2, salience,
                     segment_csr, topology_csr)
