"""Float64 CPU oracle of the bounded-activation DiT block forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``memory_bounded_video_gb300``) never imports,
links or executes anything here, and this package never imports the product
path: the two share no code.  Only the seeded input generator
(``memory_bounded_video_gb300.synth``, which holds none of the method's
arithmetic) feeds both.

Sources (web pages; cited by page title and section):

* "LayerStream: H3 Chunking" (comfy.icu node review), sections "The wall is
  activations, not weights", "How the slicing works", "The two numbers you
  set", "Where people get burned".
* "Proposal: Generic memory-aware streaming execution for transformer models"
  (ComfyUI discussion), sections "Summary", "MLP planning", the attention
  streaming plan, "Safety and fallback behavior".
* "ComfyUI-StaticPipeline", section "Four levels of chunking for long
  sequences".
* "MiniMax-H3-Comfy-NPU" article, section 2.2 (INT8 weights keep one
  ``weight_scale`` per output row).

The pages name the block's operations but never write its equations; the
readings taken where they are silent (LayerNorm with eps 1e-6 and no affine,
the order of the six modulation rows, ``(1+scale)`` modulation, the gated
residual, SwiGLU roles, no biases) are listed in the module docstring of
``oracle.block``.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (library special cases, closed forms, invariants,
brute force on tiny inputs).  No function is "parity unpinned".
"""

from .block import (  # noqa: F401
    DitWeights,
    layernorm,
    modulate,
    ln_modulate,
    mha_attention,
    silu,
    swiglu_mlp,
    dit_block,
    dit_block_chunked,
    dit_block_rows,
    final_layer,
    dequant_int8,
    block_flops,
    rms_norm,
    rope_rotate,
    lora_delta,
    merge_lora,
    qk_transform,
)
