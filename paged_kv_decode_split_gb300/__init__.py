"""Paged-KV GQA split-decode for GB300 (sm_103a).

The compute path lives in the CUDA library ``libpa.so`` (C ABI, ``include/pa.h``);
``binding`` marshals torch tensors into it.  ``workloads`` draws seeded synthetic
batches.
"""
