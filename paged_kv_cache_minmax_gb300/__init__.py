"""MinMax page selection and sparse paged GQA decode attention for GB300 (sm_103a).

The compute lives in ``libkvmm.so`` (CUDA, C ABI, declared in ``include/kvmm.h``);
:mod:`paged_kv_cache_minmax_gb300.kvmm` is its thin Python binding and
:mod:`paged_kv_cache_minmax_gb300.workloads` makes seeded synthetic inputs.
Importing this package does not load the CUDA library.
"""
