"""libstencil for GB300: 3D star-stencil sweeps and the fused acoustic wave step.

The compute path is the CUDA shared library ``libstencil.so`` (sm_103a) built from
``csrc/``; this package only marshals arguments to its C ABI. Importing the package
does not load the library; the first plan does, and fails loudly if it is missing.
"""
__all__ = ["synth", "traffic"]
