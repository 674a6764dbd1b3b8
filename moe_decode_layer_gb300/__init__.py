"""GB300 (sm_103a) small-batch MoE decode layer step behind a C ABI.

The compute lives in libmoe_decode.so (csrc/); this package builds it, exposes
its C entry points through ctypes (``_lib``), wraps a handle around torch tensors
(``layer.MoEDecodeLayer``) and draws seeded synthetic inputs (``synth``).
"""

from .synth import LayerShape, TINY, LING, MUSE_NVFP4, algorithmic_bytes  # noqa: F401


def MoEDecodeLayer(*args, **kwargs):  # noqa: N802 - thin factory, imports torch lazily
    from .layer import MoEDecodeLayer as _L
    return _L(*args, **kwargs)
