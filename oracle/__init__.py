"""CPU oracle of the DFlash speculate-and-verify step and its DDTree variant.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, fp64 restatement of
what the pages describe, written to check the GPU library against.  Only the
test suite, the package smoke check and the CPU-baseline leg of the benchmark
may import it.  The product path never calls it and shares no code with it;
the only module both sides use is ``workloads`` (seeded inputs, no method
arithmetic).

Sources (page title, then section):

* "DFlash, Diffusion LLMs, dLLM, MTP and Speculative Decoding: A Deep Research
  Report" (zhichai.net) -- "Key points" (KV injection into every draft layer,
  block_size=16 single-pass drafting), "DFlash benchmark results"
  (temperature 0, acceptance length), "Why DFlash beats EAGLE-3"
  (bidirectional block context), the MTP-vs-diffusion table.
* "DFlash speculative decoding" glossary entry (globaladvisors.biz) --
  "DFlash: architecture and workflow" (four stages: anchor, one-pass block
  draft, verification by argmax, longest accepted prefix then continue from
  the new frontier), "Mathematical view of acceptance and speedup"
  (S = C_AR / (C_DF / E[L])), "From autoregressive bottlenecks to
  speculative acceleration" (greedy AR decoding).
* "LLMs hit ludicrous speed: diffusion decoding and dMoE supercharge AI
  inference" (joindrip.ai) -- DFlash paragraph (multi-layer target hidden
  features), DDTree paragraph (draft tree from per-position distributions,
  best-first heap, ancestor-only attention mask, one target pass), and the
  tutorial paragraph (a <MASK> id appended to the vocabulary).

Modules:
  numerics  -- bf16 rounding emulation, RMSNorm, RoPE, SiLU, softmax attention
  models    -- target transformer and block-diffusion drafter, KV injection
  decode    -- greedy AR decoding, the accept rule, the DFlash loop, replay
  ddtree    -- best-first heap tree builder, ancestor masks, tree accept walk

Parity status: the transformer block composition (norm placement, SwiGLU,
GQA head mapping inside a full layer) and the draft pass (slot inputs, slot
positions, the unmasked key set, the drafter's norms) have no printed values
on the pages; they are pinned by invariants and closed-form special cases
that reduce them to textbook routines.  See the test-suite docstrings for
the pin of each function.
"""
