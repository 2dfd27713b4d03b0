"""Plain fp64 CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
link this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, tables or helpers); the
only common dependency is the seeded input generator in ``workloads.py``,
which holds none of the method's arithmetic.

What it restates, and from where:

* ``philox``  -- Philox-4x32-10, written from its published definition
  (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
  SC'11), plus the stream layout used to key every random draw.
* ``accept``  -- the acceptance / residual-resampling / bonus rule of
  "Speculative decoding internals" (tarrragon LLM notes), section
  "演算法核心：sampling 階段的接受邏輯", Steps 1-4, and the greedy rule of
  "Speculative Decoding 101" (gu-log, English), Floor 4.
* ``model``   -- a Llama-style decoder forward with no KV cache (full causal
  recompute of every position), in fp64, reading the same bf16/fp32 weight
  bits the GPU receives.
* ``generate`` -- the draft loop, verification and commit of one speculative
  step, the generation loop around it, and plain autoregressive decoding.
* ``lookup``  -- prompt-lookup (n-gram) drafting ("Speculative Decoding 101",
  Floor 6) with its one-hot proposals.
* ``quant``   -- the 4-bit group-quantized weight format (codes, bf16 scales,
  packing) and its dequantization.
* ``heads``   -- drafting by extra prediction heads on the target's own final
  hidden state ("Speculative Decoding 101", Floor 6; "Speculative decoding
  internals", 三條主流變體: MTP).

Pins that tie this oracle to something other than itself live in
``tests/test_oracle_*.py`` (worked example, exhaustive enumeration, greedy
traces, closed forms, library routines, published Philox known answers).
The forward pass is pinned only component-wise (library routines and closed
forms); the pages give no worked example of a transformer forward.
"""
