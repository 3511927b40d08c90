"""MLA chunked prefill over a paged packed-latent KV cache, for GB300 (sm_103a).

Modules
-------
``workload``  seeded synthetic inputs (numpy only).
``build``     nvcc build of the in-tree C-ABI library ``_build/libmla.so``.
``_lib``      ctypes bindings of include/mla.h.
``api``       PyTorch-facing calls (``prefill``, ``merge_states``,
              ``rope_relocate``, ``gather_latent``); importing it needs torch.

Importing this package loads nothing; the library is loaded on first use and
every call fails loudly if it is missing.
"""
