"""ctypes binding of the C ABI declared in include/moe_gb300.h.

Argument marshalling only: every step of the layer runs in the CUDA library.
Functions keep the C names; tensors may be passed as torch tensors (their
device pointer is taken) or as raw integer addresses.  Importing this module
loads the in-tree library and raises if it has not been built: there is no
fallback path.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libmoe_gb300.so")

# moe_status
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_CAPACITY = 2
MOE_ERR_BAD_ROUTE = 3
MOE_ERR_UNSUPPORTED = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_CAPACITY", 3: "MOE_ERR_BAD_ROUTE",
                4: "MOE_ERR_UNSUPPORTED", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT"}

MOE_DEV_ERR_BAD_ID = 0x1
MOE_DEV_ERR_INACTIVE_SCORE = 0x2
MOE_DEV_ERR_TIMEOUT = 0x4

MOE_BF16 = 0
MOE_MXFP8 = 1
MOE_MXFP8_1X32 = 2    # weight preparation only: 1x32 inference blocks
MOE_NVFP4 = 3         # inference only: E2M1 values, E4M3 1x16 block scales, FP32 row scales

MOE_TRAINING = 0x1
MOE_DEBUG_CHECKS = 0x2
MOE_POST_NORM = 0x4
MOE_REPLAY = 0x8
MOE_ACCUMULATE_OUT = 0x1
MOE_SAVE_INPUT_ONLY = 0x2
MOE_FUSED_LAUNCH = 0x4
MOE_ACCUMULATE_DX = 0x1
MOE_DW_FP32 = 0x2
MOE_DW_ACCUMULATE = 0x4
MOE_REPLAY_FORWARD = 0x8

# moe_saved_field
(MOE_SAVED_HEADER, MOE_SAVED_COUNTS, MOE_SAVED_OFFSETS, MOE_SAVED_POFFSETS, MOE_SAVED_PERM, MOE_SAVED_INV,
 MOE_SAVED_BLOCKS, MOE_SAVED_SCORES, MOE_SAVED_H1, MOE_SAVED_XCOL, MOE_SAVED_XCOL_SCALE, MOE_SAVED_H2COL,
 MOE_SAVED_H2COL_SCALE, MOE_SAVED_BSTART, MOE_SAVED_ROWBLOCK, MOE_SAVED_H3, MOE_SAVED_PRENORM,
 MOE_SAVED_X) = range(18)
MOE_SAVED_NUM_FIELDS = 18

# moe_buffer
(MOE_BUF_XROW, MOE_BUF_XROW_SCALE, MOE_BUF_H2ROW, MOE_BUF_H2ROW_SCALE, MOE_BUF_H3, MOE_BUF_DH3ROW,
 MOE_BUF_DH3ROW_SCALE, MOE_BUF_DH3COL, MOE_BUF_DH3COL_SCALE, MOE_BUF_DH1ROW, MOE_BUF_DH1ROW_SCALE,
 MOE_BUF_DH1COL, MOE_BUF_DH1COL_SCALE, MOE_BUF_DXR, MOE_BUF_ROUTING, MOE_BUF_ERROR, MOE_BUF_NORM,
 MOE_BUF_REPLAY, MOE_BUF_SYNC, MOE_BUF_H2F) = range(20)
MOE_BUF_NUM = 20


class moe_config(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("precision", ctypes.c_int),
                ("flags", ctypes.c_uint32), ("swiglu_limit", ctypes.c_float)]


class moe_weight(ctypes.Structure):
    _fields_ = [("precision", ctypes.c_int), ("E", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("data_t", ctypes.c_void_p),
                ("scale_t", ctypes.c_void_p)]


MOE_SLOT_MAX_LAYERS = 64


class moe_slot(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int64), ("cursor", ctypes.c_int64), ("layers", ctypes.c_int32),
                ("max_layers", ctypes.c_int32), ("offset", ctypes.c_int64 * MOE_SLOT_MAX_LAYERS),
                ("flags", ctypes.c_uint32 * MOE_SLOT_MAX_LAYERS)]


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


# Every function the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_SIGNATURES = {
    "moe_version": (ctypes.c_char_p, []),
    "moe_row_capacity": (ctypes.c_int64, [ctypes.POINTER(moe_config)]),
    "moe_saved_state_bytes": (ctypes.c_size_t, [ctypes.POINTER(moe_config)]),
    "moe_saved_state_field": (ctypes.c_int, [ctypes.POINTER(moe_config), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
    "moe_ctx_scratch_bytes": (ctypes.c_size_t, [ctypes.POINTER(moe_config)]),
    "moe_ctx_create": (ctypes.c_int, [ctypes.POINTER(moe_config), ctypes.POINTER(_P)]),
    "moe_ctx_destroy": (ctypes.c_int, [_P]),
    "moe_ctx_buffer": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "moe_ctx_get_error": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_ctx_clip_stats": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "moe_debug_copy_to_host": (ctypes.c_int, [_P, _P, ctypes.c_size_t]),
    "prepare_block_scaled_weight": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                                                   _P, _P, _P, _P, _P]),
    "moe_forward": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, _P, ctypes.POINTER(moe_weight),
                                   ctypes.POINTER(moe_weight), _P, _P, ctypes.c_uint32, _P]),
    "moe_backward": (ctypes.c_int, [_P, _P, _P, ctypes.POINTER(moe_weight), ctypes.POINTER(moe_weight), _P, _P,
                                    _P, _P, ctypes.c_uint32, _P]),
    "moe_ctx_enable_stage_timing": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_ctx_stage_times": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_float), ctypes.c_int]),
    "moe_ctx_launch_count": (ctypes.c_uint64, [_P]),
    "moe_ctx_set_max_ctas": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_ctx_test_fused_stall": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64]),
    "moe_ctx_test_tile_mode": (ctypes.c_int, [_P, ctypes.c_int]),
    "moe_ctx_set_post_norm": (ctypes.c_int, [_P, _P, ctypes.c_float]),
    "moe_post_norm_backward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "moe_weight_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_size_t)]),
    "moe_saved_input_bytes": (ctypes.c_size_t, [ctypes.POINTER(moe_config)]),
    "moe_saved_input_field": (ctypes.c_int, [ctypes.POINTER(moe_config), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
    "moe_slot_init": (ctypes.c_int, [ctypes.POINTER(moe_slot), ctypes.c_int64, ctypes.c_int32]),
    "moe_slot_push": (ctypes.c_int, [ctypes.POINTER(moe_slot), ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_uint32)]),
    "moe_slot_pop": (ctypes.c_int, [ctypes.POINTER(moe_slot), ctypes.c_int64]),
    "moe_forward_static_scratch": (ctypes.c_int, [ctypes.POINTER(moe_config), ctypes.c_int32, _P, _P, _P,
                                                  ctypes.POINTER(moe_weight), ctypes.POINTER(moe_weight), _P,
                                                  ctypes.c_uint32, _P, _P]),
}

MOE_STATIC_SCRATCH_BYTES = 64 << 20

MOE_FWD_STAGES = 5
MOE_BWD_STAGES = 6
FWD_STAGE_NAMES = ("route", "gather_x", "gemm_w13_swiglu", "gemm_w2", "combine")
BWD_STAGE_NAMES = ("gather_dh3", "gemm_w2_dgrad_swiglu_bwd", "gemm_w2_wgrad", "gemm_w13_dgrad", "gemm_w13_wgrad",
                   "reduce_dx")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run mixture_experts_routed_route_gb300.build.build())")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def _ptr(t):
    """Device/host address of a torch tensor, an int, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != MOE_OK:
        raise MoEError(fn, status)


def make_config(max_tokens, d_model, d_ff, num_experts, top_k, precision, flags=0, swiglu_limit=0.0):
    return moe_config(max_tokens, d_model, d_ff, num_experts, top_k, precision, flags, swiglu_limit)


# ------------------------------------------------------------- C functions

def moe_version():
    return LIB.moe_version().decode()


def moe_row_capacity(cfg):
    return LIB.moe_row_capacity(ctypes.byref(cfg))


def moe_saved_state_bytes(cfg):
    return LIB.moe_saved_state_bytes(ctypes.byref(cfg))


def moe_saved_state_field(cfg, field):
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    _check("moe_saved_state_field", LIB.moe_saved_state_field(ctypes.byref(cfg), field, ctypes.byref(off),
                                                              ctypes.byref(nb)))
    return off.value, nb.value


def moe_weight_bytes(precision, E, N, K, with_transpose):
    """(data, scale, data_t, scale_t) byte counts of one prepared weight."""
    out = (ctypes.c_size_t * 4)()
    _check("moe_weight_bytes", LIB.moe_weight_bytes(precision, E, N, K, int(with_transpose), out))
    return tuple(int(v) for v in out)


def moe_saved_input_bytes(cfg):
    return LIB.moe_saved_input_bytes(ctypes.byref(cfg))


def moe_saved_input_field(cfg, field):
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    _check("moe_saved_input_field", LIB.moe_saved_input_field(ctypes.byref(cfg), field, ctypes.byref(off),
                                                              ctypes.byref(nb)))
    return off.value, nb.value


def moe_slot_init(capacity, max_layers):
    """A new moe_slot of `capacity` bytes holding at most `max_layers` states."""
    slot = moe_slot()
    _check("moe_slot_init", LIB.moe_slot_init(ctypes.byref(slot), capacity, max_layers))
    return slot


def moe_slot_push(slot, full_bytes, input_bytes, remaining_layers):
    """(offset, forward call flags) of the next layer's saved state."""
    off, fl = ctypes.c_int64(), ctypes.c_uint32()
    _check("moe_slot_push", LIB.moe_slot_push(ctypes.byref(slot), full_bytes, input_bytes, remaining_layers,
                                              ctypes.byref(off), ctypes.byref(fl)))
    return off.value, fl.value


def moe_slot_pop(slot, offset):
    _check("moe_slot_pop", LIB.moe_slot_pop(ctypes.byref(slot), offset))


def moe_ctx_scratch_bytes(cfg):
    return LIB.moe_ctx_scratch_bytes(ctypes.byref(cfg))


def moe_ctx_create(cfg):
    h = ctypes.c_void_p()
    _check("moe_ctx_create", LIB.moe_ctx_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h


def moe_ctx_destroy(ctx):
    _check("moe_ctx_destroy", LIB.moe_ctx_destroy(ctx))


def moe_ctx_buffer(ctx, which):
    p, nb = ctypes.c_void_p(), ctypes.c_size_t()
    _check("moe_ctx_buffer", LIB.moe_ctx_buffer(ctx, which, ctypes.byref(p), ctypes.byref(nb)))
    return p.value, nb.value


def moe_ctx_clip_stats(ctx):
    """(clamped gate count, clamped up count) since the last call; clears them."""
    counts = (ctypes.c_uint64 * 2)()
    _check("moe_ctx_clip_stats", LIB.moe_ctx_clip_stats(ctx, counts))
    return int(counts[0]), int(counts[1])


def moe_ctx_get_error(ctx):
    bits = ctypes.c_uint32()
    _check("moe_ctx_get_error", LIB.moe_ctx_get_error(ctx, ctypes.byref(bits)))
    return bits.value


def moe_debug_copy_to_host(host_dst, dev_src, nbytes):
    _check("moe_debug_copy_to_host", LIB.moe_debug_copy_to_host(_ptr(host_dst), _ptr(dev_src), nbytes))


def prepare_block_scaled_weight(w, E, N, K, precision, data, scale, data_t, scale_t, stream=None):
    _check("prepare_block_scaled_weight",
           LIB.prepare_block_scaled_weight(_ptr(w), E, N, K, precision, _ptr(data), _ptr(scale), _ptr(data_t),
                                           _ptr(scale_t), _stream(stream)))


def moe_forward(ctx, T, x, topk_ids, topk_scores, W13, W2, out, saved=None, call_flags=0, stream=None):
    _check("moe_forward", LIB.moe_forward(ctx, T, _ptr(x), _ptr(topk_ids), _ptr(topk_scores), ctypes.byref(W13),
                                          ctypes.byref(W2), _ptr(out), _ptr(saved), call_flags, _stream(stream)))


def moe_ctx_enable_stage_timing(ctx, enable=True):
    _check("moe_ctx_enable_stage_timing", LIB.moe_ctx_enable_stage_timing(ctx, 1 if enable else 0))


def moe_ctx_stage_times(ctx, pass_):
    n = MOE_FWD_STAGES if pass_ == 0 else MOE_BWD_STAGES
    arr = (ctypes.c_float * n)()
    _check("moe_ctx_stage_times", LIB.moe_ctx_stage_times(ctx, pass_, arr, n))
    return list(arr)


def moe_ctx_launch_count(ctx):
    return LIB.moe_ctx_launch_count(ctx)


def moe_ctx_set_max_ctas(ctx, max_ctas):
    _check("moe_ctx_set_max_ctas", LIB.moe_ctx_set_max_ctas(ctx, max_ctas))


def moe_ctx_test_fused_stall(ctx, stall, wait_cycles=0):
    _check("moe_ctx_test_fused_stall", LIB.moe_ctx_test_fused_stall(ctx, int(stall), int(wait_cycles)))


def moe_ctx_test_tile_mode(ctx, mode):
    """0: row-block pairs when the capacity is dense enough, 1: row blocks, 2: pairs,
    3: the forward's pairs on CTA pairs."""
    _check("moe_ctx_test_tile_mode", LIB.moe_ctx_test_tile_mode(ctx, int(mode)))


def moe_ctx_set_post_norm(ctx, gamma, eps):
    _check("moe_ctx_set_post_norm", LIB.moe_ctx_set_post_norm(ctx, _ptr(gamma), eps))


def moe_post_norm_backward(ctx, saved, dout, dx_pre, dgamma, stream=None):
    _check("moe_post_norm_backward",
           LIB.moe_post_norm_backward(ctx, _ptr(saved), _ptr(dout), _ptr(dx_pre), _ptr(dgamma), _stream(stream)))


def moe_forward_static_scratch(cfg, T, x, topk_ids, topk_scores, W13, W2, out, device_error_word, call_flags=0,
                               stream=None):
    _check("moe_forward_static_scratch",
           LIB.moe_forward_static_scratch(ctypes.byref(cfg), T, _ptr(x), _ptr(topk_ids), _ptr(topk_scores),
                                          ctypes.byref(W13), ctypes.byref(W2), _ptr(out), call_flags,
                                          _ptr(device_error_word), _stream(stream)))


def moe_backward(ctx, saved, dout, W13, W2, dx, dW13, dW2, d_scores=None, call_flags=0, stream=None):
    _check("moe_backward", LIB.moe_backward(ctx, _ptr(saved), _ptr(dout), ctypes.byref(W13), ctypes.byref(W2),
                                            _ptr(dx), _ptr(dW13), _ptr(dW2), _ptr(d_scores), call_flags,
                                            _stream(stream)))
