"""CPU oracle for the offloaded-MoE layer forward over a GPU slot cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
CPU-baseline leg may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or runs anything here,
and this package never imports the product.  The two share no code: the only
thing both consume is the seeded data made by the input generators.

Plain, slow, obviously correct: numpy in fp64 for floating point, Python
loops where the steps are sequential, one function per step of the path:

  router.py       top-k routing with softmax renormalisation (and the tiny
                  workload's gate logits)
  distinct.py     the chunk's distinct experts as a fixed-length sorted list
  slot_cache.py   LRU slot cache with an explicit recency list: ensure()
  align.py        moe_align_block_size as a stable counting sort
  numerics.py     bf16, e2m1 and e4m3 decoding from their definitions
  expert_mlp.py   SwiGLU expert MLP over decoded weights, and the combine
  layer.py        the whole slot path and the whole-layer streamed path
  stage.py        prefill staging: non-resident runs, staged row reads

Sources (page title, section):
  FreeToken PR #676 "--moe-prefill-demand-tokens": Solution, Tests, Known
  limits, gdevenyi's review comment and the author's reply;
  gdevenyi fork PR #68 "on-demand experts for short prefills";
  vLLM fork PR #48 "Expert pool ... device-side planner": What;
  vLLM fork PR #51 follow-ups: Tests, Details.

Parity pins: every function here is checked by tests/test_oracle_*.py against
something other than itself (brute force, closed forms, invariants, hand
traces under tests/golden/).  Parity unpinned: none of the functions; the
absolute rounding of the GPU's 16-bit intermediates has no external
reference and is bounded only by the stated tolerances.
"""
