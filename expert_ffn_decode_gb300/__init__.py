"""Routed MoE-FFN step (sigmoid router, top-k, 4-bit block-quantised SwiGLU experts) on GB300.

Thin Python binding of the C ABI in ``include/moeffn.h`` (``libmoeffn.so``,
built next to this file by :mod:`expert_ffn_decode_gb300.build`). The
functions below carry the C names and only marshal arguments: every step of the
layer runs in the library's CUDA kernels. Pointer arguments accept a torch
tensor (its ``data_ptr()``), a numpy array (its host address, for
``MOE_HOST_IO``), a raw integer address, or ``None`` for NULL.

Loading fails loudly when the library has not been built; there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeffn.so")

MOE_Q4_0 = 2
MOE_Q4_1 = 3
MOE_Q4_K = 12
MOE_Q6_K = 14

MOE_ACCUMULATE = 1
MOE_RESIDUAL = 2
MOE_HOST_IO = 4
MOE_NO_PDL = 8
MOE_TRACE = 16
MOE_BATCHED = 32
MOE_F32_ACT = 64
MOE_GRAPH = 128

MOE_OK = 0
MOE_ERR_INVALID_CFG = -1
MOE_ERR_NULL_PTR = -2
MOE_ERR_ALIGNMENT = -3
MOE_ERR_UNSUPPORTED = -4
MOE_ERR_CUDA = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_WORKSPACE = -7

NORM_MIN = 6.103515625e-05  # 2^-14

# Every symbol include/moeffn.h declares.
EXPORTS = ("moe_ffn_forward", "moe_ffn_forward_ex", "moe_workspace_size", "moe_trace_offset",
           "moe_workspace_status", "moe_selftest_timeout", "moe_ffn_forward_noalloc", "moe_last_error",
           "moe_shutdown")


class moe_cfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("expert_ff", ctypes.c_int32),
        ("shared_ff", ctypes.c_int32),
        ("n_groups", ctypes.c_int32),
        ("groups_used", ctypes.c_int32),
        ("n_tokens", ctypes.c_int32),
        ("qtype", ctypes.c_int32),
        ("weights_scale", ctypes.c_float),
        ("norm_min", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("swiglu_limit", ctypes.c_float),
        ("swiglu_limit_shared", ctypes.c_float),
        ("rms_eps", ctypes.c_float),
        ("ffn_norm", ctypes.c_void_p),
        ("qtype_down", ctypes.c_int32),
    ]


def make_cfg(hidden, n_experts, top_k, expert_ff, shared_ff=0, n_groups=1, groups_used=1,
             n_tokens=1, qtype=MOE_Q4_1, weights_scale=1.0, norm_min=NORM_MIN, flags=0,
             swiglu_limit=0.0, swiglu_limit_shared=0.0, rms_eps=0.0, ffn_norm=None, qtype_down=0,
             **_ignored):
    """A :class:`moe_cfg` from keyword arguments (extra keys are ignored). ``ffn_norm`` is
    a device vector (a tensor or an address) or None; ``qtype_down`` 0 means ``qtype``."""
    return moe_cfg(hidden, n_experts, top_k, expert_ff, shared_ff, n_groups, groups_used,
                   n_tokens, qtype, weights_scale, norm_min, flags, swiglu_limit, swiglu_limit_shared,
                   rms_eps, _ptr(ffn_norm), qtype_down or 0)


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"moeffn error {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """The loaded ``libmoeffn.so`` (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m expert_ffn_decode_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, cp = ctypes.c_void_p, ctypes.POINTER(moe_cfg)
        L.moe_ffn_forward.argtypes = [vp, vp, vp, vp, vp, cp, vp]
        L.moe_ffn_forward.restype = ctypes.c_int
        L.moe_ffn_forward_ex.argtypes = [vp, vp, vp, vp, vp, cp, vp, vp, ctypes.c_size_t, vp, vp, vp]
        L.moe_ffn_forward_ex.restype = ctypes.c_int
        L.moe_workspace_size.argtypes = [cp]
        L.moe_workspace_size.restype = ctypes.c_size_t
        L.moe_trace_offset.argtypes = [cp]
        L.moe_trace_offset.restype = ctypes.c_size_t
        L.moe_workspace_status.argtypes = [vp, vp]
        L.moe_workspace_status.restype = ctypes.c_int
        L.moe_selftest_timeout.argtypes = [vp, vp]
        L.moe_selftest_timeout.restype = ctypes.c_int
        L.moe_ffn_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, cp, vp, vp]
        L.moe_ffn_forward_noalloc.restype = ctypes.c_int
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_shutdown.argtypes = []
        L.moe_shutdown.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(obj):
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if hasattr(obj, "data_ptr"):
        return obj.data_ptr()
    if hasattr(obj, "ctypes"):
        return obj.ctypes.data
    raise TypeError(f"cannot pass {type(obj).__name__} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def moe_ffn_forward(x, router_w, router_bias, expert_blocks, shared_blocks, cfg, out):
    return lib().moe_ffn_forward(_ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(expert_blocks),
                                 _ptr(shared_blocks), ctypes.byref(cfg), _ptr(out))


def moe_ffn_forward_ex(x, router_w, router_bias, expert_blocks, shared_blocks, cfg, out, workspace,
                       workspace_bytes, stream, topk_ids=None, topk_w=None):
    return lib().moe_ffn_forward_ex(_ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(expert_blocks),
                                    _ptr(shared_blocks), ctypes.byref(cfg), _ptr(out), _ptr(workspace),
                                    int(workspace_bytes), _stream(stream), _ptr(topk_ids), _ptr(topk_w))


def moe_workspace_size(cfg):
    return lib().moe_workspace_size(ctypes.byref(cfg))


def moe_trace_offset(cfg):
    return lib().moe_trace_offset(ctypes.byref(cfg))


# Names of the MOE_TRACE timeline points, in order.
TRACE_POINTS = ("router_start", "router_x_ready", "router_done", "gate_up_sel_keys",
                "gate_up_start", "gate_up_x_quantised", "gate_up_waited", "gate_up_picked", "gate_up_rows_landed",
                "gate_up_end", "gate_up_dots", "gate_up_sums",
                "down_start", "down_picked", "down_rows_requested", "down_waited", "down_act_staged",
                "down_rows_landed", "down_end", "gate_up_sel_cands", "down_loop_done", "down_sums",
                "gate_up_sel_ranked")
TRACE_STRIDE = 24  # u64 words per CTA


def moe_workspace_status(workspace, stream=None):
    return lib().moe_workspace_status(_ptr(workspace), _stream(stream))


def moe_selftest_timeout(workspace, stream=None):
    return lib().moe_selftest_timeout(_ptr(workspace), _stream(stream))


def moe_ffn_forward_noalloc(x, router_w, router_bias, expert_blocks, shared_blocks, cfg, out, stream=None):
    """The step without any allocation (fixed 512 KiB device scratch; blocking)."""
    return lib().moe_ffn_forward_noalloc(_ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(expert_blocks),
                                         _ptr(shared_blocks), ctypes.byref(cfg), _ptr(out), _stream(stream))


def moe_last_error():
    return lib().moe_last_error().decode()


def moe_shutdown():
    return lib().moe_shutdown()


def check(rc):
    """Raise :class:`MoeError` with the library's message when ``rc`` is an error."""
    if rc != MOE_OK:
        raise MoeError(rc, moe_last_error())
    return rc
