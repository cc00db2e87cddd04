"""GB300-native fused weight-quantized SwiGLU expansion.

    hidden = silu(x . Wg^T) * (x . Wu^T)

x is a bf16 [M, H] activation; Wg and Wu are [I, H] matrices in affine group
quantisation (w = scale * q + bias per group of gs consecutive K elements, q an
unsigned 4- or 8-bit code packed little-endian into uint32 words, bf16 scales
and biases).  All arithmetic runs in the CUDA kernels of ``libqswiglu.so``
behind the C ABI in ``include/qswiglu.h``; the Python binding in ``ops.py``
only marshals torch tensors into that ABI.

Importing this package does not load the CUDA library; the first call into
``quantized_swiglu_mlp_gb300.ops`` does, and raises if it is missing.
"""

__all__ = ["ops", "inputs"]


def __getattr__(name):
    if name in ("ops", "inputs", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
