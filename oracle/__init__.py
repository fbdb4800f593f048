"""The oracle: a plain, slow, fp64 CPU statement of what the hot path computes.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
anything here; only the tests, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline / reference arm do.  The oracle shares no code with the CUDA
library: its only common dependency is the seeded input generator ``synth``.

Modules
-------
``beam``  batched beam search step, finished set, stopping rules, finalisation
          (pages: "Transformers中的Beam Search高效实现" and "9.2 贪心搜索与束搜索").
``bpd``   blockwise parallel decoding: predict, verify, accept, and the greedy
          decoder it must reproduce ("Blockwise Parallel Decoding for Deep
          Autoregressive Models", §2-§4).
``kv``    KV-cache reorder: the naive gather and a paged block table with
          copy-on-write ("9.2 贪心搜索与束搜索", §9.2.2 and §9.2.4).

Pinning status: every function here is pinned by a ``-m "not gpu"`` test against
values the pages print, closed forms, brute force on tiny inputs or a library
routine, except where a docstring says "parity unpinned".
"""
