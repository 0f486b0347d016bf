"""CPU oracle for the tensor-parallel Qwen3-style forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, links or
calls anything under ``oracle/``; only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg use it.  It shares no code with the CUDA
path.

* ``oracle.forward``  -- the unsharded reference forward (plain definitions,
  float64 by default), and the vocab-parallel / tensor-parallel emulation that
  builds rank shards with its own index maps and sums rank partials with a
  counted "all-reduce".
* ``oracle.brute``    -- scalar pure-Python loops for tiny shapes, written
  independently of ``oracle.forward`` (no BLAS, no torch), used to pin it.

Sources ("the pages"):
  [TP]   ai-infra-handbooks, "Tensor parallelism from scratch": sections
         "Two ways to split", "Implementation" (tp.py), "KV heads and the
         limit on TP".
  [SHD]  jaehun.me, "mini-sglang 08: How several ranks share one ledger":
         section "Weights are cut by name" (python/minisgl/models/weight.py:
         13-14, 34-52) and python/minisgl/layers/linear.py:102-106.
  [CH9]  zero-to-sglang, "Chapter 9 Multi-process and Tensor Parallelism",
         section 3.3 "Loading Weights and Model State" (shard then merge,
         VocabParallelEmbedding, ParallelLMHead).

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (closed forms, library routines, brute force,
the numbers printed in [TP]).  No function is left "parity unpinned".
"""
