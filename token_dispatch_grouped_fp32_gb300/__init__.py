"""GB300-native (sm_103a) forward pass of one mixture-of-experts layer.

- ``moe``    : binding of libmoe (include/moe.h) -- route, dispatch, grouped
               SwiGLU experts, combine, and the fused forward.
- ``synth``  : seeded synthetic inputs of the benchmark workloads.
- ``build``  : in-tree build of libmoe.so with nvcc for sm_103a.

``import token_dispatch_grouped_fp32_gb300.moe`` loads the CUDA library and
fails loudly if it has not been built.
"""
