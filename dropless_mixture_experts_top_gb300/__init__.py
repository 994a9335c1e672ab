"""GB300-native dropless mixture-of-experts expert layer (training forward + backward).

The compute path is a C-ABI CUDA library (``include/moe.h``) built for sm_103a;
``moe`` is its thin ctypes binding and ``synth`` draws seeded synthetic inputs.
Import the binding explicitly: ``from dropless_mixture_experts_top_gb300 import moe``.
"""
