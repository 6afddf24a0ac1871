"""CPU oracle for the heterogeneous-batch LoRA delta -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import anything here.  The product path never does: the CUDA library
shares no code with this package, and this package imports nothing from the
product package.

Contents
  pool.py   the page allocator, per-adapter page tables, the adapter "load"
            into pool pages, and the token grouping (segments) -- in plain
            Python/numpy, following the policy stated in each docstring.
  lora.py   ctypes front end of oracle.c, the fp64 loop implementation of
            y += s (x A) B that gathers every weight element through the
            page table.
  ref.py    the dense brute force (numpy fp64 matmul) used to pin oracle.c.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (brute force, closed forms, invariants, library routines).
"""
