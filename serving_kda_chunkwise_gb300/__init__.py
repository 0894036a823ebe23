"""GB300-native Kimi Delta Attention (KDA): chunked forward, decode step and gate.

The compute lives in ``libkda.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/kda.h``).  ``serving_kda_chunkwise_gb300.kda`` is the thin
Python binding with the same entry-point names; importing it loads the library
and fails loudly if it has not been built (there is no fallback path).
"""

__all__ = ["kda", "inputs"]


def __getattr__(name):
    if name == "kda":
        from . import kda as _k
        return _k
    if name == "inputs":
        from . import inputs as _i
        return _i
    raise AttributeError(name)
