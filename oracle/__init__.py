"""CPU oracle for the DSV3-style MXFP8 MoE layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 numpy statement of what the layer computes, written from
the Mixture-of-Kittens write-ups (Cursor blog summary, iThome/techlab report,
mlqm commentary) and the plain readings they leave open. Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it. It shares no code with the CUDA path (``moe_layer_dsv3_gb300``)
and imports nothing from it; the only common module is ``gen``, which draws
inputs and holds none of the layer's arithmetic.

Modules:
  mxfp8     E4M3 codec and MX block quantisation (OCP MX v1.0 reading of "MXFP8")
  sigmoid   the specified fp32 sigmoid both sides implement independently
  route     router logits, group-limited top-k on sigmoid+bias, gate normalisation
  schedule  per-expert counts, prefix sums, stable ranks, ring laps/slots
  layer     expert SwiGLU FFN, shared expert, combine, full backward
  waves     the SM-wave token threshold heuristic of the commentary

Every function here has a pin in ``tests/test_oracle_*.py``; none is
"parity unpinned".
"""
