"""GB300-native (sm_103a) deterministic routed SwiGLU expert layer, forward and backward.

The compute path is the C-ABI library ``libmok.so`` (hand-written CUDA, see ``include/mok.h``);
``mixture_experts_layer_build_gb300.mok`` is its thin Python binding.  Importing this package
does not load the library; importing ``.mok`` does, and fails loudly when it is missing.
"""
__version__ = "0.1.0"
