"""GB300-native packed BitLinear products (i2_s, TQ2_0, W1A8).

The compute runs in the CUDA library ``libbl.so`` (C ABI, see include/bl.h).
``gemm_bl_gemv_gb300.binding`` is the thin Python layer over it; importing this
package does not load the library, so the input generators in ``synth`` can be
used on machines without a GPU.
"""
import importlib

__all__ = ["binding", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
