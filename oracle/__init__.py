"""CPU oracle for the MoE decode layer-step with a cross-token prerouter.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or executes
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code with the CUDA
library: it does its own bf16 rounding, its own nibble packing and unpacking and its
own routing; it receives the same seeded input arrays as the CUDA path and nothing
else.

Everything is plain numpy in float64 (weights are dequantised exactly into fp64,
activations arrive as bf16 bit patterns and are widened exactly).  Sources, by page
title and section:

* "The Other Half of the Memory Wall" (Edge0), §3.1 "Problem" / "Executor paths" /
  "Math contract": int4 affine group-64 expert weights with per-group scale and bias,
  nine stacked tensors per layer, expert math down(silu(gate(x)) * up(x)).
* same page, §3.2 "Head": fc1 -> erf-GELU -> fc2 plus a linear residual path, input
  feature = [hidden ; one-hot of this layer's routing at this token ; one-hot at the
  previous token].  §3.2 "Prediction-as-routing": the prediction is the routing.
* same page, §3.3: unmerged recovery LoRA y = W_int4(x) + (alpha/r) * B A x.
* same page, Appendix A "Softmax-topk": g = softmax(l), inds = top-k(g, K),
  w = g[inds] / sum_inds g; and "Sigmoid-group": group scores from the top-2 sigmoids,
  top groups kept, top-k within them, w = s * sigma / (sum sigma + 1e-20).
* BigMoeOnEdge "Route-ahead" notes: layer L's selection is its own gate ranked on the
  hidden state N layers earlier in the same forward pass.

Modules:
  ``bf16``     bfloat16 <-> float conversion (round to nearest even).
  ``int4``     affine group-64 packing, unpacking and dequantisation.
  ``routing``  softmax-top-k with renormalisation; sigmoid-group routing; the gap a
               routing decision rests on.
  ``layer``    router, prerouter head, SwiGLU expert, LoRA linear, layer-step,
               prefill chunk and one decode token through a stack (head-routed,
               own-gate and route-ahead layers).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, textbook values, brute force or page-printed numbers; none is
"parity unpinned".
"""
