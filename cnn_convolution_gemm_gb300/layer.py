"""Torch-facing convenience over the C ABI: a conv layer that owns its
descriptor, packed weights and workspace as torch CUDA tensors.

Memory and streams come from PyTorch; every computation is a call into
libgbconv.so through ``binding``.
"""
from __future__ import annotations

import torch

from . import binding as B

TORCH_DTYPE = {B.CONV_BF16: torch.bfloat16, B.CONV_F32: torch.float32, B.CONV_INT8: torch.int8}


def current_stream_handle() -> int:
    return torch.cuda.current_stream().cuda_stream


class ConvLayer:
    """One convolution: y = act(conv(x, w) + bias (+ residual)).

    NHWC activations [N][H][W][C], weights [K][R][S][C/groups] (NCHW / [K][C/g][R][S]
    for the fp32 NCHW layout)."""

    def __init__(self, N, C, H, W, K, R, S, stride=1, pad=0, dilation=1, groups=1,
                 dtype=B.CONV_BF16, layout=B.CONV_NHWC, act=B.CONV_ACT_NONE,
                 has_residual=False, scale=None, input_shuffle=1):
        self.shape = (N, C, H, W, K, R, S, stride, pad, dilation, groups)
        self.dtype, self.layout = dtype, layout
        self.desc = B.conv_desc_create(N, C, H, W, K, R, S, stride, pad, dilation, groups, dtype)
        if layout != B.CONV_NHWC:
            B.conv_desc_set_layout(self.desc, layout)
        if act or has_residual:
            B.conv_desc_set_epilogue(self.desc, act, has_residual)
        if input_shuffle > 1:
            B.conv_desc_set_input_shuffle(self.desc, input_shuffle)
        self.scale = scale
        if scale is not None:
            B.conv_desc_set_requant(self.desc, scale.data_ptr())
        self.OH, self.OW = B.conv_desc_get_output_dims(self.desc)
        self.algo = None
        self.wpack = None
        self.ws = None

    def __del__(self):
        d = getattr(self, "desc", None)
        if d is not None:
            try:
                B.conv_desc_destroy(d)
            except Exception:
                pass

    @property
    def output_shape(self):
        N, K = self.shape[0], self.shape[4]
        if self.layout == B.CONV_NHWC:
            return (N, self.OH, self.OW, K)
        if self.layout == B.CONV_NC32HW32:
            return (N, K // 32, self.OH, self.OW, 32)
        return (N, K, self.OH, self.OW)

    def applicable_algos(self):
        out = []
        for i in range(B.conv_algo_count(self.desc)):
            a, name, ok = B.conv_algo_info(self.desc, i)
            if ok:
                out.append((a, name))
        return out

    def fastrun(self, stream=None):
        """Fast-Run selection for this layer's shape; returns (algo, times_ms)."""
        return B.conv_fastrun_select(self.desc, current_stream_handle() if stream is None else stream)

    def prepack(self, w: torch.Tensor, algo: int = B.CONV_ALGO_AUTO, stream=None):
        a = B.conv_algo_resolve(self.desc) if algo == B.CONV_ALGO_AUTO else algo
        nbytes = B.conv_weights_packed_size(self.desc, a)
        wpack = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=w.device)
        B.conv_weights_prepack(self.desc, a, w.data_ptr(), wpack.data_ptr(),
                               current_stream_handle() if stream is None else stream)
        wsb = B.conv_workspace_size(self.desc, a)
        self.ws = torch.empty(wsb, dtype=torch.uint8, device=w.device) if wsb else None
        self.wpack, self.algo = wpack, a
        return a

    def forward(self, x: torch.Tensor, bias=None, residual=None, out=None, stream=None):
        if self.wpack is None:
            raise RuntimeError("prepack() the weights first")
        if out is None:
            out = torch.empty(self.output_shape, dtype=x.dtype, device=x.device)
        ws = self.ws
        B.conv_fwd(self.desc, x.data_ptr(), self.wpack.data_ptr(),
                   None if bias is None else bias.data_ptr(),
                   None if residual is None else residual.data_ptr(), out.data_ptr(), self.algo,
                   None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(),
                   current_stream_handle() if stream is None else stream)
        return out

    __call__ = forward

    def forward_host(self, x_host: torch.Tensor, bias=None, residual_host=None, out_host=None,
                     n_chunk=0, stream=None):
        """The same forward pass on host tensors (x, residual, y page-locked in host
        memory; weights and bias on the device): the batch runs in chunks of
        n_chunk images whose copies overlap the convolution (conv_fwd_host).
        Stream-ordered: out_host is complete once the stream has caught up."""
        if self.wpack is None:
            raise RuntimeError("prepack() the weights first")
        if out_host is None:
            out_host = torch.empty(self.output_shape, dtype=x_host.dtype).pin_memory()
        need = B.conv_fwd_host_scratch_size(self.desc, self.algo, n_chunk)
        sc = getattr(self, "_host_scratch", None)
        if sc is None or sc.numel() < need:
            dev = self.wpack.device
            sc = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            self._host_scratch = sc
        B.conv_fwd_host(self.desc, x_host.data_ptr(), self.wpack.data_ptr(),
                        None if bias is None else bias.data_ptr(),
                        None if residual_host is None else residual_host.data_ptr(),
                        out_host.data_ptr(), self.algo, n_chunk, sc.data_ptr(), sc.numel(),
                        current_stream_handle() if stream is None else stream)
        return out_host
