"""GB300 (sm_103a) ternary linear layer: CUDA kernels behind a C ABI (include/tl.h).

Submodules:
  tl     ctypes binding of the C ABI plus the TernaryLinear convenience class
  build  compiles csrc/*.cu into libtl_gb300.so in this directory
  synth  seeded synthetic inputs (no layer arithmetic)
The binding is imported lazily so that `synth` and `build` work without torch
or a built library.
"""

__all__ = ["tl", "build", "synth"]


def __getattr__(name):
    if name in __all__:
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
