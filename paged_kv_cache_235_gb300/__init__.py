"""tfpa: paged GQA attention over a 256-position page pool, for GB300 (sm_103a).

The compute path is the C-ABI library ``libtfpa.so`` built from ``csrc/``;
``binding`` is a thin ctypes layer over it with the same entry-point names.
"""

__all__ = ["binding", "workloads"]
