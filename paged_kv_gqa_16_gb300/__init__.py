"""paged_kv_gqa_16_gb300 -- paged GQA decode attention for one GB300 (sm_103a).

The compute lives in ``libpkv.so`` (hand-written CUDA, C ABI declared in
``include/pkv.h``).  ``paged_kv_gqa_16_gb300.pkv`` is the thin ctypes binding
with the same entry-point names; ``workloads`` draws seeded synthetic inputs.
Importing the package does not load the library; the first call does, and it
raises if the library is missing rather than computing anything elsewhere.
"""

__all__ = ["pkv", "workloads"]
