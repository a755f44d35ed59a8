"""Plain, slow, fp64 CPU oracle for the speculative-decoding verification pass.

TEST INFRASTRUCTURE ONLY.  This package exists to check the CUDA library
against the mathematics the pages define.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product path (the C-ABI library and
its Python binding) never imports, links or executes anything here, and this
package imports nothing from the product package.

Modules
-------
accept   -- temperature / nucleus distribution, the ratio test, residual
            resampling, bonus token, greedy rule, inverse-CDF draw.
model    -- the Llama-style decoder forward over the gamma+1 new positions
            (RMSNorm, RoPE, GQA attention over a bf16 KV cache, SwiGLU,
            LM head) and the KV rollback rule.
weights  -- the seeded synthetic weights: Philox4x64-10 counter-based
            generator + Box-Muller in fp64, rounded to bf16.
bf16     -- round-to-nearest-even conversion of fp64 values to bf16.
tree     -- draft-tree verification: ancestor masks and depths, the tree
            forward, the per-node acceptance walk, the KV commit.
constrain -- constrained acceptance: one allowed-token mask applied to the
            target and draft logits alike.
gamma    -- the dynamic speculation-depth controller (rolling acceptance
            window, depth maximising expected tokens per millisecond).

Every function cites the passage it follows.  Parity status per function:

* accept.*                     pinned (worked example, exact enumeration,
                               chi-square, alpha, E[tokens], greedy rule;
                               draft_sample against torch's softmax, its
                               draws by chi-square, its T = 0 argmax)
* model.rmsnorm/rope/attention pinned against torch library routines and
  /swiglu/lm_head              mathematical invariants (lm_head: torch's
                               linear, identity and one-hot heads, linearity)
* model.forward                pinned by invariants only (one pass equals
                               sequential passes; rollback then re-verify
                               equals a fresh pass; sublayers pinned above).
                               The pages print no logits, so end-to-end
                               values are otherwise unpinned.
* weights                      pinned by the published Philox4x64-10
                               known-answer vectors and normal moments.
* tree.*                       pinned (the printed mask / depths and
                               expected-depth values, simulated coins, chain
                               equivalence, path-by-path chain passes,
                               chi-square of the walk's output)
* gamma.*                      pinned (printed expected-token values,
                               simulated coins, simulated throughput per
                               depth, limits, the page's alpha < 0.65
                               statement, window and warm-up)
* constrain.apply_mask         pinned (restricted-softmax closed form,
                               chi-square and acceptance rate with the same
                               mask on both sides, one-sided mask breaks it)
"""
