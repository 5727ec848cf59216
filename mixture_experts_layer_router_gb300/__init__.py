"""LatentMoE layer forward for GB300 (sm_103a).

``capi`` binds the C-ABI library (``include/latentmoe.h``) with ctypes;
``synth`` draws seeded synthetic inputs. Importing the package does not load
the library; ``capi.load()`` does, and fails loudly when it is missing.
"""
