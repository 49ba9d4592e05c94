"""GB300-native GPT-2 124M cached decode step (cachedStep), its full-prefix
twin (infer) and the int8 group-64 variant, as hand-written sm_103a CUDA
kernels behind a C ABI (include/gpt2.h, libgpt2gb.so).

``stream_decode_gb300.gpt2`` is the Python binding (it loads the library and
fails loudly if it is missing); ``stream_decode_gb300.synth`` draws seeded
synthetic checkpoints and token ids; ``stream_decode_gb300.build`` compiles
the library.
"""
