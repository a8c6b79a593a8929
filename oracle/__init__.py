"""CPU oracle for paged KV-cache attention (TEST INFRASTRUCTURE ONLY).

A plain, slow, obviously correct restatement of what the paged decode path
computes, written from the PagedAttention pages (the apxml course page
"PagedAttention Memory Management", the katajob Q&A "What problem does
PagedAttention solve for the KV cache in vLLM?", the foundry page on paged block
allocation for the KV cache, and the "PagedAttention, clearly explained"
thread).  Arithmetic is fp64 except where the stored format fixes a precision
(the fp32 product before the E4M3 rounding of a quantised slot write).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  It shares no code with the CUDA
library in ``paged_kv_cache_137_gb300/`` and imports nothing from it; the only
common module is ``workloads`` (seeded random inputs, no method arithmetic).

Modules
    sizing     block bytes, pool capacity, blocks per sequence, waste
    allocator  free-block stack, block tables, reference counts, fork, CoW
    e4m3       OCP E4M3 (FN) encode/decode
    pool       the physical K/V pool: slot writes and block copies
    attention  decode attention gathered through block tables
    prefill    multi-query (prefill) causal attention through block tables
    prefix_cache  block allocator with prefix caching (published full blocks)
    preemption    preemption by recompute, watermark admission
    scenario   the five synthetic workloads built with the pieces above

Parity pins: every function is checked in ``tests/test_oracle_*.py`` against
values the pages print, closed forms, brute force and library routines; none
is unpinned.
"""
from . import sizing, allocator, e4m3, pool, attention, prefill, prefix_cache, preemption  # noqa: F401
