"""libsp: shared-prefix, prefill-only label readout for GB300 (sm_103a).

``prefill_only_shared_gb300.sp`` is the ctypes binding of the C-ABI library
``libsp.so`` (built in-tree by ``prefill_only_shared_gb300.build``);
``prefill_only_shared_gb300.workloads`` draws seeded synthetic inputs.
"""
