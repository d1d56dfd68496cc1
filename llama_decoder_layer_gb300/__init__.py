"""GB300 (sm_103a) Llama decoder-layer forward over a paged KV cache.

``binding`` wraps the C ABI of ``libllama_layer.so`` (include/llama_layer.h);
``inputs`` draws the seeded synthetic workloads; ``build`` compiles the
library.  The library is loaded on first use and there is no fallback path.
"""
