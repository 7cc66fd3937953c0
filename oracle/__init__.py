"""CPU oracle for one MoE-transformer decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The GPU product path never calls it and shares no
code with it; the two meet only in the seeded input generator (``synth``).

The oracle is the plain definition of the step the decode megakernel computes
(pages: "Cohere Publishes One-Kernel Server for North Mini Code" — "The delay
is between operations" (normalization, projections, attention, routing);
"Inside the Megakernel Serving Engine" (QKV, then attention, then MoE); "Cohere
fuses an entire decode step into one GPU program" (project query and key,
attention, routing network)).  The megakernel reorders and tiles this work;
it must reach the same result up to rounding.

Precision: bf16 weights are widened exactly and all arithmetic is float64.
Two places turn floating point into integers; both decide on float32-rounded
values, the kernel's precision: the router's top-k and the greedy argmax.
The only rounding the method itself performs, bf16 storage of the new
token's K and V in the paged cache, is reproduced exactly (``bf16_rne``).

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against closed forms, brute force on tiny inputs, library routines
(``torch.nn.functional.rms_norm``, float32->bf16 conversion) and invariants
(key-order permutation, zero-branch reductions, single-expert = dense FFN).
Whole-model values with random weights have no printed counterpart on the
pages: beyond those pins, end-to-end values are "parity unpinned".
"""
from .decode import (  # noqa: F401
    bf16_rne, rmsnorm, rope, gqa_attention, route, silu, expert_ffn,
    OracleRequest, LayerTrace, StepResult, attention_block, moe_block, decode_layer, lm_head,
    decode_step,
)
