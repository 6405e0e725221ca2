"""GB300 (sm_103a) convolution backward-data: dx = dgrad(dy, w) as a
stride-decomposed implicit GEMM, behind a C ABI (include/conv_bwd_data.h).

Modules:
  binding    ctypes binding of the C ABI (loads lib/libconv_bwd_data.so; raises
             if it is missing -- there is no CPU fallback)
  build      in-tree nvcc build of the library
  workloads  seeded synthetic inputs and the named problem shapes

``binding`` is imported lazily so that the input generators stay usable on
machines where the CUDA library has not been built.
"""

__all__ = ["binding", "build", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
