"""GB300 (sm_103a) persistent MoE decode megakernel.

One decode step of an MoE transformer runs as one persistent kernel: one CTA
per SM walks a host-prepared list of tile tasks whose readiness is tracked by
counters in global memory.  The C ABI lives in ``libmk.so`` (``include/mk.h``);
``persistent_moe_decode_02_gb300.mk`` is its thin Python binding.
"""
