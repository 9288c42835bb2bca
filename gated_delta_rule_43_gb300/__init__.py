"""GB300-native Kimi Delta Attention (KDA): chunked prefill and decode.

The compute lives in ``libkda.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/kda.h``); ``gated_delta_rule_43_gb300.kda`` is the thin
Python binding and ``gated_delta_rule_43_gb300.inputs`` draws seeded
synthetic workloads.  The binding loads the library lazily and raises if it
is missing: there is no CPU fallback.
"""
__all__ = ["inputs", "kda"]
