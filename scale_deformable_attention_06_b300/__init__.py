"""Multi-scale deformable attention (MSDeformAttn) core for NVIDIA B300.

The computation runs in libmsda.so (hand-written CUDA for sm_103a, C ABI in
include/msda.h); this package is its Python binding.  See _capi for the call
signatures: msda_forward, msda_forward_fused, msda_backward,
msda_backward_fused, and the 3-D variant msda3d_forward, msda3d_backward.
MSDeformAttnFunction, MSDeformAttnFusedFunction and MSDeformAttn3DFunction
pair each forward call with its backward call for torch.autograd.
"""
from ._capi import (EXPORTED, LIBRARY, MSDA_ACCUMULATE_GRAD_VALUE, MSDA_BF16, MSDA_DETERMINISTIC, MSDA_F32,
                    MSDA_OPT_ALIGN_CORNERS, MSDA_OPT_PER_LEVEL_SOFTMAX, MSDAError, lib, msda_backward, msda_backward_fused, msda_backward_noalloc,
                    msda_backward_workspace_size, msda_forward, msda_forward_fused, msda_problem, msda3d_backward,
                    msda3d_forward)
from ._autograd import MSDeformAttn3DFunction, MSDeformAttnFunction, MSDeformAttnFusedFunction

__all__ = ["msda_forward", "msda_forward_fused", "msda_backward", "msda_backward_fused", "msda3d_forward",
           "msda3d_backward",
           "msda_backward_workspace_size", "msda_backward_noalloc", "MSDAError",
           "MSDA_DETERMINISTIC", "MSDA_ACCUMULATE_GRAD_VALUE", "MSDA_F32", "MSDA_BF16",
           "MSDA_OPT_PER_LEVEL_SOFTMAX", "MSDA_OPT_ALIGN_CORNERS", "LIBRARY", "EXPORTED",
           "lib", "msda_problem", "MSDeformAttnFunction", "MSDeformAttnFusedFunction", "MSDeformAttn3DFunction"]
