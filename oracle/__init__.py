"""Plain, slow CPU oracle for the shared-prefix classifier path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs use it.  It shares no code, tables or helpers
with the CUDA library; it consumes the same seeded input tensors and nothing
else.

Everything is computed from the plain definition, in float64 with numpy:

* ``staging``       -- token trie, segments, node-token layout and the staged
                       submission rounds (LLM2Jev "shared prefix" page,
                       section on staged submission for a cold request).
* ``attention``     -- every branch's full token sequence recomputed on its
                       own with naive causal softmax attention (no sharing).
* ``readout``       -- full-vocabulary log-softmax at the branch's last
                       position, gathered at the requested label ids
                       (openjev-sglang article, prefill-only readout section).
* ``label_softmax`` -- stable softmax renormalisation of the label logprobs
                       and the argmax label (same article, worked yes/no
                       example).
* ``postprocess``   -- question-type readouts and the confidence value
                       (same article, sections on confidence and on the three
                       question types).
* ``cache``         -- the radix prefix cache across calls (LLM2Jev page,
                       section on reusing the radix cache).
* ``batching``      -- the admission rule of continuous batching across
                       requests (openjev-multimodal performance page, next
                       steps).
* ``options``       -- multi-token option scores (chain-rule sums of
                       readout log-probabilities) and label-prior calibration
                       (openjev-multimodal performance page, next steps).

Parity status of every function is stated in its module docstring; all are
pinned by tests under ``tests/`` marked ``not gpu``.
"""
