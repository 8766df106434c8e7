"""Torch-facing wrapper of the C ABI: device buffers come from torch, every
computation runs in the CUDA library.

``PreparedWeight`` holds one stacked expert weight in the form the GEMMs read
(``prepare_block_scaled_weight``); ``MoELayer`` owns one context and offers
``forward`` / ``backward`` on torch tensors; ``ActivationSlot`` packs several
layers' saved states into one buffer and decides which of them keep only
their input (``moe_slot_*``).
"""

import numpy as np
import torch

from . import abi

_DT = {"bf16": abi.MOE_BF16, "mxfp8": abi.MOE_MXFP8, "mxfp8_1x32": abi.MOE_MXFP8_1X32, "nvfp4": abi.MOE_NVFP4}


def precision_code(precision):
    return _DT[precision] if isinstance(precision, str) else int(precision)


class PreparedWeight:
    """One stacked weight [E, N, K] prepared for the GEMMs.

    BF16: ``data`` is the caller's tensor, ``data_t`` its transpose
    [E, K, N] (for the input-gradient GEMMs).  MXFP8: E4M3 codes with one
    E8M0 scale per 32x32 tile, in both orientations (the transposed codes
    too unless mn_major).  "mxfp8_1x32": forward only, one scale per 1x32
    block of a row along K.  "nvfp4": inference only, E2M1 codes and E4M3
    scales per 16 values along K in 128-row x 64-value chunks (``data``)
    and one FP32 scale per row (``scale``)."""

    def __init__(self, w, precision, with_transpose=True, stream=None, mn_major=False):
        """mn_major (MXFP8 with_transpose): keep only the input-gradient scale
        atoms; the input-gradient GEMMs then read the forward codes MN-major
        instead of a transposed copy (E*N*K bytes less)."""
        assert w.dtype == torch.bfloat16 and w.is_cuda and w.dim() == 3
        w = w.contiguous()
        self.precision = precision_code(precision)
        E, N, K = w.shape
        self.shape = (E, N, K)
        dev = w.device
        self.data_t = self.scale = self.scale_t = None
        if self.precision == abi.MOE_NVFP4:
            nbytes = abi.moe_weight_bytes(self.precision, E, N, K, False)
            self.data = torch.empty(nbytes[0], dtype=torch.uint8, device=dev)
            self.scale = torch.empty(E * N, dtype=torch.float32, device=dev)
            abi.prepare_block_scaled_weight(w, E, N, K, self.precision, self.data, self.scale, None, None, stream)
        elif self.precision == abi.MOE_MXFP8_1X32:
            self.data = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
            self.scale = torch.empty(E * N * (K // 32) + 16, dtype=torch.uint8, device=dev)
            abi.prepare_block_scaled_weight(w, E, N, K, self.precision, self.data, self.scale, None, None, stream)
        elif self.precision == abi.MOE_MXFP8:
            self.data = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
            self.scale = torch.empty(E * N * (K // 32) + 16, dtype=torch.uint8, device=dev)
            if with_transpose:
                if not mn_major:
                    self.data_t = torch.empty((E, K, N), dtype=torch.uint8, device=dev)
                self.scale_t = torch.empty(E * K * (N // 32) + 16, dtype=torch.uint8, device=dev)
            abi.prepare_block_scaled_weight(w, E, N, K, self.precision, self.data, self.scale, self.data_t,
                                            self.scale_t, stream)
        else:
            self.data = w
            if with_transpose:
                self.data_t = torch.empty((E, K, N), dtype=torch.bfloat16, device=dev)
                abi.prepare_block_scaled_weight(w, E, N, K, self.precision, None, None, self.data_t, None, stream)
        self.struct = abi.moe_weight(self.precision, E, N, K, abi._ptr(self.data), abi._ptr(self.scale),
                                     abi._ptr(self.data_t), abi._ptr(self.scale_t))


class MoELayer:
    """One routed MoE layer bound to a context (fixed scratch)."""

    def __init__(self, max_tokens, d_model, d_ff, num_experts, top_k, precision, training=False, debug=False,
                 device="cuda", swiglu_limit=0.0, post_norm=False, replay=False):
        flags = ((abi.MOE_TRAINING if training else 0) | (abi.MOE_DEBUG_CHECKS if debug else 0)
                 | (abi.MOE_POST_NORM if post_norm else 0) | (abi.MOE_REPLAY if replay else 0))
        self.cfg = abi.make_config(max_tokens, d_model, d_ff, num_experts, top_k, precision_code(precision), flags,
                                   swiglu_limit)
        self.device = torch.device(device)
        self.D, self.F, self.E, self.K = d_model, d_ff, num_experts, top_k
        self.training = training
        self.ctx = abi.moe_ctx_create(self.cfg)
        self.r_cap = abi.moe_row_capacity(self.cfg)

    def close(self):
        if self.ctx is not None:
            torch.cuda.synchronize(self.device)
            abi.moe_ctx_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------- state
    def new_saved(self, input_only=False):
        nb = abi.moe_saved_input_bytes(self.cfg) if input_only else abi.moe_saved_state_bytes(self.cfg)
        return torch.empty(nb, dtype=torch.uint8, device=self.device)

    def saved_field(self, saved, field, dtype, shape, input_only=False):
        off, nb = (abi.moe_saved_input_field if input_only else abi.moe_saved_state_field)(self.cfg, field)
        esz = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        assert n * esz <= nb
        return saved[off:off + n * esz].view(dtype).view(*shape)

    def read_buffer(self, which, dtype, shape):
        """Copy one scratch region to host memory (tests only)."""
        ptr, nb = abi.moe_ctx_buffer(self.ctx, which)
        out = np.empty(shape, dtype=dtype)
        assert out.nbytes <= nb
        abi.moe_debug_copy_to_host(out.ctypes.data, ptr, out.nbytes)
        return out

    def error_bits(self):
        return abi.moe_ctx_get_error(self.ctx)

    def clip_stats(self):
        return abi.moe_ctx_clip_stats(self.ctx)

    def set_post_norm(self, gamma, eps):
        """gamma: bf16 [D] on the device, kept referenced while the layer uses it."""
        abi.moe_ctx_set_post_norm(self.ctx, gamma, eps)
        self._gamma = gamma

    def post_norm_backward(self, saved, dout, dx_pre=None, dgamma=None, stream=None):
        """dout = dL/d(normalised output) -> (dL/d(pre-norm output), dL/dgamma)."""
        T = dout.shape[0]
        if dx_pre is None:
            dx_pre = torch.empty((T, self.D), dtype=torch.bfloat16, device=self.device)
        if dgamma is None:
            dgamma = torch.empty((self.D,), dtype=torch.float32, device=self.device)
        abi.moe_post_norm_backward(self.ctx, saved, dout, dx_pre, dgamma, stream)
        return dx_pre, dgamma

    # ----------------------------------------------------------- compute
    def forward(self, x, ids, scores, W13, W2, out=None, saved=None, accumulate=False, save_input_only=False,
                fused=False, stream=None):
        """fused: the whole inference forward as one launch (MOE_FUSED_LAUNCH)."""
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.D), dtype=torch.bfloat16, device=self.device)
        flags = ((abi.MOE_ACCUMULATE_OUT if accumulate else 0) | (abi.MOE_SAVE_INPUT_ONLY if save_input_only else 0)
                 | (abi.MOE_FUSED_LAUNCH if fused else 0))
        abi.moe_forward(self.ctx, T, x, ids, scores, W13.struct, W2.struct, out, saved, flags, stream)
        return out

    def backward(self, saved, dout, W13, W2, dx=None, dW13=None, dW2=None, accumulate_dx=False, dw_fp32=False,
                 dw_accumulate=False, d_scores=None, replay=False, stream=None):
        T = dout.shape[0]
        dt = torch.float32 if dw_fp32 else torch.bfloat16
        if dx is None:
            dx = torch.empty((T, self.D), dtype=torch.bfloat16, device=self.device)
        if dW13 is None:
            dW13 = torch.empty((self.E, 2 * self.F, self.D), dtype=dt, device=self.device)
        if dW2 is None:
            dW2 = torch.empty((self.E, self.D, self.F), dtype=dt, device=self.device)
        flags = ((abi.MOE_ACCUMULATE_DX if accumulate_dx else 0) | (abi.MOE_DW_FP32 if dw_fp32 else 0)
                 | (abi.MOE_DW_ACCUMULATE if dw_accumulate else 0) | (abi.MOE_REPLAY_FORWARD if replay else 0))
        abi.moe_backward(self.ctx, saved, dout, W13.struct, W2.struct, dx, dW13, dW2, d_scores, flags, stream)
        return dx, dW13, dW2


class ActivationSlot:
    """One device buffer of `capacity` bytes holding the saved states of a
    stack of layers ("Dist-MoE: Speed-of-light distributed Mixture-of-Experts
    kernels", section 04 "Activation Packing and Dynamic Recompute").
    ``push`` gives the next layer its state (a view of the buffer) and tells
    whether it keeps only its input; ``pop`` returns it, in reverse order."""

    def __init__(self, capacity, max_layers=abi.MOE_SLOT_MAX_LAYERS, device="cuda"):
        self.buf = torch.empty(capacity, dtype=torch.uint8, device=device)
        self.slot = abi.moe_slot_init(capacity, max_layers)

    def push(self, layer, remaining_layers):
        """(saved view, input_only) for `layer`, with `remaining_layers`
        layers of the same size still to come after it in this slot."""
        full, inp = abi.moe_saved_state_bytes(layer.cfg), abi.moe_saved_input_bytes(layer.cfg)
        off, flags = abi.moe_slot_push(self.slot, full, inp, remaining_layers)
        input_only = bool(flags & abi.MOE_SAVE_INPUT_ONLY)
        return self.buf[off:off + (inp if input_only else full)], input_only

    def pop(self, saved):
        abi.moe_slot_pop(self.slot, saved.data_ptr() - self.buf.data_ptr())
