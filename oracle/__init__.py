"""Plain CPU oracle for the hybrid sliding-window two-pool KV scheme.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It is a slow, direct restatement of what the source pages define, written in
numpy / plain Python with float64 arithmetic for attention:

* ``allocator``  - free-page ledgers, the full->SWA mapping, alloc / alloc_extend
                   / alloc_decode, free / free_swa, out-of-window eviction.
* ``attention``  - key sets of sliding / chunked-local / full layers and
                   brute-force softmax with a per-head sink logit and GQA.
* ``sizing``     - the two-pool sizing rule.
* ``codecs``     - bf16 and FP8-E4M3 encoders/decoders (store dtype = bytes).
* ``envelope``   - page-major envelope addressing (kernel-facing row ids).
* ``hitrule``    - the W-contiguous-non-tombstone prefix-hit rule.
* ``kvstore``    - per-layer / envelope KV pools that store and gather rows.
* ``radix``      - the SWA component of the radix prefix cache.
* ``unified``    - the unified FULL/SWA pool allocated from both ends of one
                   page range, with its virtual-to-physical page tables.

Source pages (cited by title and section throughout):
  [SWA note]      "SWA in SGLang" design note (zdszero.github.io/swa.html)
  [Pools 15]      "SGLang source teardown (15): memory pools and allocators"
                  (pinghaoyang.com.cn)
  [PR 34602]      "Unified pool MHA/SWA -> dense per-layer views", SGLang PR
                  #34602 summary (prhub.com.cn)

The oracle shares no code with the CUDA path and imports nothing from it.
"""
