"""Topology-scheduled sparse attention on GB300 (sm_103a).

The product is the C-ABI library libtsa.so (include/tsa.h); this package builds it and binds
its three operations with the same names:

* ``tsa_build_schedule``      -- causal CSR block schedule from K (sink, local window, top-k
                                 by elder-rule salience over key-block centroids);
* ``tsa_dense_causal_csr``    -- the dense causal CSR;
* ``tsa_scheduled_attention`` -- causal attention over a CSR block schedule.
"""
from .binding import (STATUS_NAMES, TSA_BF16, TSA_F16, TsaError, lib, library_path,  # noqa: F401
                      tsa_build_schedule, tsa_build_schedule_workspace_bytes, tsa_dense_causal_csr,
                      tsa_last_device_status, tsa_schedule_max_nnz, tsa_scheduled_attention)
