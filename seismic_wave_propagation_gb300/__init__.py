"""libstencil for GB300: 3D star-stencil sweeps and the fused acoustic wave step.

The compute path is the CUDA shared library ``libstencil.so`` (sm_103a) built from
``csrc/``; this package only marshals arguments to its C ABI (``StencilPlan`` mirrors
``stencil_plan_create`` / ``stencil_apply`` / ``wave_step`` / ``stencil_plan_status``).
Importing the package does not load the library; the first plan does, and raises if it
has not been built.
"""
from ._lib import (KIND_APPLY, KIND_SEMI, KIND_WAVE, KIND_WAVE_PML, StencilError, StencilPlan,  # noqa: F401
                   StencilSlabs, last_error, load, version)
from . import synth, traffic  # noqa: F401

__all__ = ["StencilPlan", "StencilSlabs", "StencilError", "KIND_APPLY", "KIND_WAVE", "KIND_WAVE_PML", "KIND_SEMI", "load", "last_error",
           "version", "synth", "traffic"]
