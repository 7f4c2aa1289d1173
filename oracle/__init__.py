"""Plain CPU oracle for compressed-KV-cache attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.

The oracle restates, slowly and in the plainest form, what the method
computes.  Sources (web pages on the subject):

* "MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative
  KV Cache" (pith.science review page and its verdict JSON, arXiv 2411.18077):
  2-bit asymmetric quantisation with FP16 scale and zero-point, keys grouped
  per channel and values per token, 16 INT2 codes per INT32 word, heavy
  hitters chosen once at the end of prefill from cumulative attention scores
  plus a recent window, pyramid per-layer budgets, a two-pass prefill kernel
  whose second pass emits column-wise cumulative attention scores, and a
  128-token full-precision residual buffer.
* "DiffKV" verdict JSON (arXiv 2412.03131), fields ``key_machinery`` and the
  referee report's Algorithm 1 comments: significance = mean attention a
  token receives from later tokens, max over the GQA group, compared with
  alpha_h/N and alpha_l/N to choose K8V4, K4V2 or pruning as a token leaves
  the recent window.
* "Don't Discard, but Keep It Small" (MiKV rebuttal page): important tokens
  at high precision, the rest at low precision, nothing evicted, high to low
  re-quantisation as importance drops, precision groups stored contiguously
  because attention is permutation invariant after positional encoding.

Arithmetic rules: attention and softmax in float64; the quantiser follows
one fixed float32 operation sequence (see ``oracle.quant``) so that codes
are reproducible bit for bit.  numpy never contracts a*b+c into an FMA, so
every float32 step below is one IEEE round-to-nearest operation.

Modules: ``quant`` (quantise / pack / dequantise), ``attention`` (prefill
pass 1 and 2, decode attention), ``select`` (budgets, heavy hitters + recent
window), ``policies`` (the MiniKV, DiffKV and MiKV cache life cycles),
``accounting`` (cache byte counts).

Parity status of every function is listed in its docstring; functions whose
result the pages fix nowhere are marked "parity unpinned".
"""
