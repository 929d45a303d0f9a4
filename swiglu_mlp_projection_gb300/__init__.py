"""GB300-native fused SwiGLU up-projection: h = silu(x.W_gate) (.) (x.W_up).

The compute path is the CUDA library built from ``csrc/`` (a C ABI declared in
``include/swiglu.h``); this package only marshals arguments into it.  The
library is loaded on first use and its absence is an error: there is no CPU
fallback.
"""
