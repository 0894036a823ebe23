"""GB300-native Kimi Delta Attention (KDA): chunked forward, decode step and gate.

The compute lives in ``libkda.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/kda.h``).  ``serving_kda_chunkwise_gb300.kda`` is the thin
Python binding with the same entry-point names; importing it loads the library
and fails loudly if it has not been built (there is no fallback path).
Submodules are imported explicitly (``from serving_kda_chunkwise_gb300 import kda``)
so that importing the package itself never touches the library.
"""
