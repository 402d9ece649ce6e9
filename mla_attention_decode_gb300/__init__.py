"""GB300-native single-token MLA decode.

The product is ``libmla_decode.so`` (C ABI, hand-written sm_103a CUDA kernels);
``mla_attention_decode_gb300.binding`` is the thin Python marshalling layer over
it and ``mla_attention_decode_gb300.synth`` draws seeded synthetic inputs.
Importing this package does not load the CUDA library; the binding loads it on
first use and raises if it is missing.
"""
__all__ = ["binding", "synth"]
