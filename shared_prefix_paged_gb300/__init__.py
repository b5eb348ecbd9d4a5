"""Cascade attention over a shared-prefix paged KV cache, native to GB300 (sm_103a).

The compute lives in a C-ABI shared library built from ``csrc/`` (see
``include/csp.h``); ``csp`` is the thin ctypes binding over it.  Importing this
package loads nothing: the library is opened on first use of ``csp``, and a
missing library is an error, never a fallback.
"""

__all__ = ["csp", "workloads", "accounting"]
