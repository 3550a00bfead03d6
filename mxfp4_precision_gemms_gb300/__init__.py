"""GB300-native H16/H32 + MXFP4 linear-layer GEMMs (sm_103a).

The compute path lives in ``libmxfp4.so`` (hand-written CUDA kernels behind a C ABI,
``include/mxfp4.h``); ``binding`` marshals torch tensors through ctypes, and
``linear.mxfp4_linear`` wires the Fprop / Dgrad / Wgrad calls into torch autograd.
"""
