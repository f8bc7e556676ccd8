"""GB300-native Mixture-of-Experts layer (router top-k, layout, pull dispatch,
MXFP8/BF16 grouped SwiGLU FFN, deterministic weighted combine, backward).

The compute path is the C-ABI CUDA library ``libmok.so`` (sm_103a); the Python
side here only marshals arguments to it (``combine_top_routing_gb300.mok``).
"""
