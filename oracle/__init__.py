"""Float64 CPU oracle for paged-KV decode attention and KV-append.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain statement of what
the CUDA path must compute, written from the source pages and nothing else.
It shares no code with ``paged_kv_cache_222_gb300`` (no kernels, headers,
helpers, tables or constants) and neither side imports the other.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs
of ``bench.py`` may import it; the product path never does.

Sources (web pages, cited by title and section throughout):

* [FN]  FactNode, "Sub-Millisecond Token Scheduling: Inside Disaggregated
        KV-Cache Paging for Frontier LLMs".
* [SC]  systemcraft.online lesson "LLM inference: prefill, decode, KV cache"
        (course c03).
* [UI]  ultrainstinct.tech, "Architecting Multi-Tier Disaggregated KV-Cache
        Hierarchies for Terabyte-Scale LLM Inference".

Modules:

* ``formats``          bf16 / fp32 / FP8-E4M3 encodings from their definitions.
* ``paged_attention``  block-table walk, decode attention, KV append.
* ``footprint``        KV-cache footprint formula and the capacity arithmetic.

Every function here is pinned by ``-m "not gpu"`` tests against something
other than itself (printed values from the pages, closed forms, invariants,
library routines on special cases, brute force on tiny inputs).
"""

from . import formats, paged_attention, footprint  # noqa: F401
