"""CPU oracle for greedy speculative decoding — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the speculative step
computes, in float64 on the CPU with plain PyTorch CPU ops. It exists to check
the CUDA path, and only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import it. The product
path never calls it and shares no code with it: the only common module is
``synth`` (seeded input generation, none of the method's arithmetic).

Sources it follows (page title, then the section):
  * "I Got 28 TPS Out of Free Kaggle GPUs. Here's What It Took." (dev.to):
    "Speculative Decoding: The Idea" (draft guesses K tokens, the target checks
    all of them in one pass, the agreed tokens are committed) and "Why It Kept
    Breaking (and How I Fixed It)" (static cache, explicit positions, in-place
    rewind of the KV cache to the last accepted position).
  * "Qwen3.5-397B on 20 GPUs, through a relay" (Sangama results):
    "Speculative decoding: correct, but slower (for now)" (look-back n-gram
    guesses of up to 4 tokens from the last 2-4 tokens; the verifier returns
    its own choice at every position; speculative output equals normal
    greedy decoding token for token).
The pages give no model equations. The transformer forward follows the
architecture the workloads name (Qwen2-style GQA + RoPE + RMSNorm + SwiGLU);
every such choice is marked "reading" in the function that makes it.

Modules:
  model   -- fp64 forward of one decoder over a KV cache (rows independent)
  decode  -- greedy decoding, acceptance, in-place rollback, n-gram lookup and
             the speculative loop
  nf4     -- NormalFloat-4 codebook, blockwise quantisation, dequantisation
"""
