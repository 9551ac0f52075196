"""learnable_scale_fake_gb300: learnable-scale fake-quant (QDQ forward, straight-
through scale gradient, per-head observer) as hand-written CUDA for GB300
(sm_103a), behind the C ABI of include/aqfq.h.

``aqfq`` is the ctypes binding of libaqfq.so; ``synth`` draws the seeded
synthetic inputs.  Importing the package loads nothing: the CUDA library is
loaded on the first call and raises if it is missing.
"""
__all__ = ["aqfq", "synth"]
