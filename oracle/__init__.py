"""fp64 CPU oracle for the n-gram speculative-decoding hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the GPU library computes.  Only the test suite, the
``smoke()`` check of ``__graft_entry__`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product path
(the CUDA library and its Python binding) never imports, calls or links
anything here, and this package never imports the product.

Sources (the pages this restates, by title and section):

* "AX Engine: An LLM Inference Engine Built Exclusively for Apple Silicon
  M4+", section "Core Technical Architecture & Methods": bigram/trigram
  tables built at runtime, up to 4 draft tokens per step, validation by the
  target forward, EMA acceptance gate (tau = 0.1, threshold = 0.5), O(1)
  rollback by moving the sequence-length pointer; section "Supported Model
  Families" (table): Gemma's logit soft cap.
* "SwiftLM: Apple Silicon native MLX Swift LLM inference server", the
  paragraph on algorithmic equivalence (Leviathan et al.): accept a draft
  with probability P_target / P_draft, resample from the corrected
  distribution on rejection; the M1 Ultra benchmark paragraph: repetition
  penalty 1.1, temperature 0.6; the DFlash warning paragraph: pure greedy
  (argmax) verification as the temperature-0 special case.

Modules
-------
``philox``  counter-based Philox4x32-10 (Salmon et al., SC'11) and the maps
            from its words to uniforms and Gumbel noise.
``verify``  row transform, softmax, accept test, residual / bonus sampling,
            epilogue (token write-back, kv_len rollback, EMA gate).
``ngram``   bigram/trigram continuation statistics and chained drafting.

Every function states the passage it follows.  Parity status of each part
is recorded in the module docstrings ("pinned by" lines name the tests).
"""
