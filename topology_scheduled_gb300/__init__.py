"""Topology-scheduled sparse attention on GB300 (sm_103a).

The product is the C-ABI library libtsa.so (include/tsa.h); this package builds it and binds
its operations with the same names:

* ``tsa_build_schedule``      -- causal CSR block schedule from K (sink, local window, top-k
                                 by elder-rule salience over key-block centroids), with the
                                 elder rule's ties broken by block index or centroid content;
* ``tsa_dense_causal_csr``    -- the dense causal CSR;
* ``tsa_fixed_segment_csr`` / ``tsa_segment_csr`` -- the CSR of a segment mask;
* ``tsa_scheduled_attention`` -- causal attention over a CSR block schedule
  (``tsa_scheduled_attention_fwd`` also returns the row log-sum-exp);
* ``tsa_scheduled_attention_backward`` -- its dQ, dK, dV;
* ``tsa_block_sums`` / ``tsa_build_schedule_from_sums`` -- the build in two halves, for keys
  whose lanes are spread over several GPUs (``distributed.build_schedule_lane_sharded``);
* ``tsa_topology_attention_host`` -- one forward step (schedule + attention) from host
  tensors, the host<->device copies overlapped with the work.
"""
from .binding import (STATUS_NAMES, TIE_RULES, TSA_BF16, TSA_F16, TsaError, lib,  # noqa: F401
                      library_path, tsa_build_schedule, tsa_build_schedule_workspace_bytes,
                      tsa_dense_causal_csr, tsa_fixed_segment_csr, tsa_fixed_segment_nnz,
                      tsa_last_device_status, tsa_schedule_max_nnz, tsa_scheduled_attention,
                      tsa_scheduled_attention_fwd, tsa_scheduled_attention_backward,
                      tsa_attention_backward_workspace_bytes, tsa_segment_csr, tsa_block_sums,
                      tsa_build_schedule_from_sums, tsa_topology_attention_host,
                      tsa_debug_set_wait_injection)
