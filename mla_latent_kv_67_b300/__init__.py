"""B300-native absorbed, paged MLA decode.

The CUDA library (``libmla_b300.so``, built from ``csrc/``) is loaded lazily by
:mod:`mla_latent_kv_67_b300.binding`; importing this package alone does not
touch the GPU.
"""
__all__ = ["synth", "binding"]
