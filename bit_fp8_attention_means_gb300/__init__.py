"""VC-Attention hot path for one GB300 (sm_103a).

FP8 non-causal attention with V-Smooth (k-means grouping, joint K/V gather,
block-mean residual quantization, in-softmax mean restore) and ExpCast-FP8,
as hand-written CUDA kernels behind the C ABI in ``include/vc.h``.
``vc`` is the ctypes binding; ``inputs`` draws the seeded synthetic workloads;
``schedule`` drives the amortized denoising schedule.  Importing the package
does not load the CUDA library; the first call does, and raises if it is
missing.
"""
from .vc import (VcError, VcShape, alloc_quantized, shape_of, vc_attn_fwd, vc_cluster,  # noqa: F401
                 vc_quantize)
