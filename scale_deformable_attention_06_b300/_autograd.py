"""torch.autograd bindings of the MSDeformAttn calls.

Each Function's forward is the library's forward call and its backward the
matching backward call, so a model can train through the sampler the way the
Deformable DETR and deformable-attention tutorial pages describe it: the value
branch, the sampling locations (or the reference points and offsets) and the
attention weights (or logits) all receive gradients ("可变形 DETR：加速收敛的稀疏
注意力检测器" §3.3; "可变形注意力：多尺度稀疏采样与视觉检测实战解析" §2.2-§2.3).
Argument marshalling only: both directions run in libmsda.so.

spatial_shapes and level_start_index take no gradient.  grad_value comes out
of the library in fp32 and is handed to autograd in the dtype of value (bf16
values get a bf16 gradient, as autograd requires).  `flags` is passed to the
backward call (MSDA_DETERMINISTIC for run-to-run identical gradients) less
MSDA_ACCUMULATE_GRAD_VALUE: autograd sums gradients into .grad itself;
`options` goes to both calls.
"""
import torch

from . import _capi


def _grad_out(grad_output, value):
    return grad_output.to(value.dtype).contiguous()


def _backward_flags(flags):
    return flags & ~_capi.MSDA_ACCUMULATE_GRAD_VALUE


class MSDeformAttnFunction(torch.autograd.Function):
    """out [N, Len_q, M*D] = msda_forward(value, spatial_shapes,
    level_start_index, sampling_locations, attention_weights); the backward
    gives value, sampling_locations and attention_weights their gradients
    through msda_backward."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, sampling_locations, attention_weights, flags=0,
                options=0):
        out = _capi.msda_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                                 options=options)
        ctx.save_for_backward(value, sampling_locations, attention_weights)
        ctx.levels = (spatial_shapes, level_start_index)
        ctx.flags, ctx.options = _backward_flags(flags), options
        return out

    @staticmethod
    def backward(ctx, grad_output):
        value, loc, attn = ctx.saved_tensors
        gv, gl, ga = _capi.msda_backward(value, *ctx.levels, loc, attn, _grad_out(grad_output, value),
                                         flags=ctx.flags, options=ctx.options)
        return gv.to(value.dtype), None, None, gl, ga, None, None


class MSDeformAttnFusedFunction(torch.autograd.Function):
    """out = msda_forward_fused(value, spatial_shapes, level_start_index,
    reference_points, sampling_offsets, attention_logits): the locations and
    the softmax formed in the kernel; the backward gives value,
    reference_points, sampling_offsets and attention_logits their gradients
    through msda_backward_fused."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, reference_points, sampling_offsets, attention_logits,
                flags=0, options=0):
        out = _capi.msda_forward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                                       attention_logits, options=options)
        ctx.save_for_backward(value, reference_points, sampling_offsets, attention_logits)
        ctx.levels = (spatial_shapes, level_start_index)
        ctx.flags, ctx.options = _backward_flags(flags), options
        return out

    @staticmethod
    def backward(ctx, grad_output):
        value, ref, off, logits = ctx.saved_tensors
        gv, gref, goff, glog = _capi.msda_backward_fused(value, *ctx.levels, ref, off, logits,
                                                          _grad_out(grad_output, value), flags=ctx.flags,
                                                          options=ctx.options)
        return gv.to(value.dtype), None, None, gref, goff, glog, None, None


class MSDeformAttn3DFunction(torch.autograd.Function):
    """The trilinear variant: out = msda3d_forward(value, spatial_shapes
    [L, 3] as (frames, H, W), level_start_index, sampling_locations
    [N, Len_q, M, L, K, 3], attention_weights); gradients through
    msda3d_backward."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, sampling_locations, attention_weights, flags=0,
                options=0):
        out = _capi.msda3d_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                                   options=options)
        ctx.save_for_backward(value, sampling_locations, attention_weights)
        ctx.levels = (spatial_shapes, level_start_index)
        ctx.flags, ctx.options = _backward_flags(flags), options
        return out

    @staticmethod
    def backward(ctx, grad_output):
        value, loc, attn = ctx.saved_tensors
        gv, gl, ga = _capi.msda3d_backward(value, *ctx.levels, loc, attn, _grad_out(grad_output, value),
                                           flags=ctx.flags, options=ctx.options)
        return gv.to(value.dtype), None, None, gl, ga, None, None
