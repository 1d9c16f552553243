"""Plain, slow CPU oracle of the expert-slot-cache MoE layer (TEST INFRASTRUCTURE).

This package is the reference the CUDA library is checked against.  It is
test infrastructure only: nothing but ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  The product path
(``serving_layer_moe_gb300``) never imports it and has no CPU fallback.

It shares no code with the CUDA path.  It is written from the four web pages
that describe the FreeToken MoE serving engine:

  * "FreeToken: treat the whole PC as one" (signalovernoise.tech newsletter)
  * "FreeToken, or why your laptop was never the bottleneck" (snackonai.com deep dive)
  * "FreeToken: a 753B model on one GPU, and the two bandwidths that decide
    everything" (ai.thesatyajit.com article)
  * "FreeToken runs frontier-scale MoE models by treating the whole PC as the
    inference platform" (dev.to summary)

Modules:
  formats       exact decoding of f32 / bf16 / e4m3 (+128x128 block scales),
                NVFP4 and MXFP4
  policy        the miss split q* and its clamps, branch times
  cache         list-based global LRU of (layer, expert) slots: decode control,
                full-layer prefill residency, resize
  ffn           SwiGLU expert in float64 and the fixed-order combine
  static_split  the static placement comparators: routing-blind split and
                prefill-pinned hot subset

Every function says which passage it follows.  Readings of passages the
pages leave open are listed with the function that takes them.
"""
