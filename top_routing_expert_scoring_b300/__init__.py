"""Python binding of the B300 MoE layer forward library (libmoe_b300.so).

Argument marshalling only: every function forwards to the C entry point of the same name in
include/moe_b300.h, passing tensors as device pointers and the current CUDA stream.  Tensors
are allocated by the caller (torch is used for device memory and streams only).  Importing
this package fails with ImportError when the compiled library is missing; there is no other
code path.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MoeConfig", "MoeError", "make_config", "lib", "lib_path", "workspace", "capacity",
    "workspace_size", "check_config", "sync_status", "status_string", "version",
    "moe_router_topk", "moe_aux_stats", "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_ffn", "moe_shared_ffn",
    "moe_combine", "moe_expert_choice", "moe_forward", "moe_forward_timed", "moe_workspace_views",
    "moe_workspace_views_ec",
    "moe_selftest_timeout", "EXPORTED", "SCORE", "ROUTING", "DTYPE",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libmoe_b300.so")

if not os.path.exists(lib_path):
    raise ImportError(
        f"{lib_path} is missing: build it with `python top_routing_expert_scoring_b300/build.py` "
        "(needs nvcc with sm_103a support)")

lib = ctypes.CDLL(lib_path)

SCORE = {"softmax": 0, "sigmoid": 1}
ROUTING = {"token_choice": 0, "expert_choice": 1}
DTYPE = {"bf16": 0, "f32": 1}


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("E", ctypes.c_int32),
        ("k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
        ("score", ctypes.c_int32), ("routing", ctypes.c_int32), ("n_groups", ctypes.c_int32),
        ("topk_groups", ctypes.c_int32), ("renormalize", ctypes.c_int32),
        ("route_scale", ctypes.c_float), ("capacity_factor", ctypes.c_float),
        ("dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
    ]

    def __repr__(self):
        return "MoeConfig(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status}: {status_string(status)}")


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoeConfig)
_I32P = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "moe_version": ([], ctypes.c_char_p),
    "moe_check_config": ([_CFG], ctypes.c_int),
    "moe_capacity": ([_CFG, _I32P], ctypes.c_int),
    "moe_workspace_size": ([_CFG, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "moe_sync_status": ([_P, _P], ctypes.c_int),
    "moe_router_topk": ([_CFG, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_aux_stats": ([_CFG, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_dispatch": ([_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_dispatch_noalloc": ([_CFG] + [_P] * 12, ctypes.c_int),
    "moe_expert_ffn": ([_CFG, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_shared_ffn": ([_CFG, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_combine": ([_CFG, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_expert_choice": ([_CFG, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_forward": ([_CFG] + [_P] * 17, ctypes.c_int),
    "moe_forward_timed": ([_CFG] + [_P] * 19, ctypes.c_int),
    "moe_workspace_views": ([_CFG, _P] + [ctypes.POINTER(_P)] * 5, ctypes.c_int),
    "moe_workspace_views_ec": ([_CFG, _P] + [ctypes.POINTER(_P)] * 4, ctypes.c_int),
    "moe_selftest_timeout": ([_P, ctypes.c_int32, _P], ctypes.c_int),
    "moe_router_backward_workspace_size": ([_CFG, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "moe_router_backward": ([_CFG] + [_P] * 6 + [ctypes.c_float, ctypes.c_float] + [_P] * 5,
                            ctypes.c_int),
    "moe_bias_update": ([_CFG, _P, _P, ctypes.c_float, _P], ctypes.c_int),
    "moe_quantize_fp8": ([ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P], ctypes.c_int),
    "moe_fp8_workspace_size": ([_CFG, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "moe_forward_fp8": ([_CFG] + [_P] * 21, ctypes.c_int),
}
EXPORTED = tuple(_SIGS)

for _name, (_args, _ret) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _ret


def status_string(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def version() -> str:
    return lib.moe_version().decode()


def make_config(T, d_model, E, k, d_ff, d_ff_shared=0, score="softmax",
                routing="token_choice", n_groups=1, topk_groups=None, renormalize=True,
                route_scale=1.0, capacity_factor=0.0, dtype="bf16", out_dtype="f32") -> MoeConfig:
    """out_dtype: "f32" returns the fp32-accumulated layer output as is; "bf16" rounds it."""
    return MoeConfig(int(T), int(d_model), int(E), int(k), int(d_ff), int(d_ff_shared),
                     SCORE[score], ROUTING[routing], int(n_groups),
                     int(n_groups if topk_groups is None else topk_groups), int(bool(renormalize)),
                     float(route_scale), float(capacity_factor), DTYPE[dtype], DTYPE[out_dtype])


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (the library reads device memory only)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, status):
    if status != 0:
        raise MoeError(name, status)


def check_config(cfg: MoeConfig) -> int:
    return lib.moe_check_config(ctypes.byref(cfg))


def capacity(cfg: MoeConfig) -> int:
    c = ctypes.c_int32()
    _check("moe_capacity", lib.moe_capacity(ctypes.byref(cfg), ctypes.byref(c)))
    return c.value


def workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size", lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def workspace(cfg: MoeConfig, device="cuda"):
    """A zeroed device workspace of moe_workspace_size() bytes (torch allocation)."""
    import torch
    return torch.zeros(workspace_size(cfg), dtype=torch.uint8, device=device)


def sync_status(ws, stream=None) -> int:
    return lib.moe_sync_status(_ptr(ws), _stream(stream))


def moe_router_topk(cfg, x, w_gate, bias, logits, topk_idx, topk_w, ws, stream=None):
    _check("moe_router_topk", lib.moe_router_topk(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(logits), _ptr(topk_idx),
        _ptr(topk_w), _ptr(ws), _stream(stream)))


def moe_aux_stats(cfg, logits, topk_idx, f, P, l_balance, z_loss, ws, stream=None):
    _check("moe_aux_stats", lib.moe_aux_stats(
        ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(f), _ptr(P), _ptr(l_balance),
        _ptr(z_loss), _ptr(ws), _stream(stream)))


def moe_dispatch(cfg, topk_idx, x, counts, kept, offsets, pos, row_of, perm, x_perm, n_dropped,
                 ws, stream=None):
    _check("moe_dispatch", lib.moe_dispatch(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(kept), _ptr(offsets),
        _ptr(pos), _ptr(row_of), _ptr(perm), _ptr(x_perm), _ptr(n_dropped), _ptr(ws),
        _stream(stream)))


def moe_dispatch_noalloc(cfg, topk_idx, x, counts, kept, offsets, pos, row_of, perm, x_perm,
                         n_dropped, status, stream=None):
    """moe_dispatch without a workspace, for callers that may not allocate device memory (the
    scratch is a fixed array inside the library; T <= 65536, E <= 256).  status: int32[2] on
    the device, (code, detail) of the first device-side error."""
    _check("moe_dispatch_noalloc", lib.moe_dispatch_noalloc(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(kept), _ptr(offsets),
        _ptr(pos), _ptr(row_of), _ptr(perm), _ptr(x_perm), _ptr(n_dropped), _ptr(status),
        _stream(stream)))


def moe_expert_ffn(cfg, x_perm, offsets, w13, w2, y_perm, ws, stream=None):
    _check("moe_expert_ffn", lib.moe_expert_ffn(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(w2), _ptr(y_perm),
        _ptr(ws), _stream(stream)))


def moe_shared_ffn(cfg, x, ws13, ws2, shared_out, ws, stream=None):
    _check("moe_shared_ffn", lib.moe_shared_ffn(
        ctypes.byref(cfg), _ptr(x), _ptr(ws13), _ptr(ws2), _ptr(shared_out), _ptr(ws),
        _stream(stream)))


def moe_combine(cfg, y_perm, row_of, topk_w, shared_out, out, stream=None):
    _check("moe_combine", lib.moe_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(row_of), _ptr(topk_w), _ptr(shared_out), _ptr(out),
        _stream(stream)))


def moe_expert_choice(cfg, logits, ec_tokens, ec_w, tok_ptr, tok_rows, ws, stream=None):
    _check("moe_expert_choice", lib.moe_expert_choice(
        ctypes.byref(cfg), _ptr(logits), _ptr(ec_tokens), _ptr(ec_w), _ptr(tok_ptr),
        _ptr(tok_rows), _ptr(ws), _stream(stream)))


def moe_forward(cfg, x, w_gate, bias, w13, w2, ws13, ws2, out, topk_idx=None, topk_w=None,
                f=None, P=None, l_balance=None, z_loss=None, n_dropped=None, ws=None,
                stream=None):
    _check("moe_forward", lib.moe_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(w13), _ptr(w2), _ptr(ws13),
        _ptr(ws2), _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(f), _ptr(P), _ptr(l_balance),
        _ptr(z_loss), _ptr(n_dropped), _ptr(ws), _stream(stream)))


def moe_forward_timed(cfg, x, w_gate, bias, w13, w2, ws13, ws2, out, topk_idx=None, topk_w=None,
                      f=None, P=None, l_balance=None, z_loss=None, n_dropped=None, ws=None,
                      stream=None, ev_begin=None, ev_end=None):
    """moe_forward plus two torch.cuda.Event (enable_timing) recorded around the expert GEMMs."""
    _check("moe_forward_timed", lib.moe_forward_timed(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(w13), _ptr(w2), _ptr(ws13),
        _ptr(ws2), _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(f), _ptr(P), _ptr(l_balance),
        _ptr(z_loss), _ptr(n_dropped), _ptr(ws), _stream(stream), ev_begin.cuda_event,
        ev_end.cuda_event))


def moe_workspace_views(cfg, ws):
    """Device addresses (ints) of logits, row_of, offsets, x_perm, y_perm inside ws."""
    outs = [ctypes.c_void_p() for _ in range(5)]
    _check("moe_workspace_views", lib.moe_workspace_views(
        ctypes.byref(cfg), _ptr(ws), *[ctypes.byref(o) for o in outs]))
    return [o.value for o in outs]


def moe_workspace_views_ec(cfg, ws):
    """Device addresses (ints) of ec_tokens, ec_w, tok_ptr, tok_rows inside ws (expert
    choice)."""
    outs = [ctypes.c_void_p() for _ in range(4)]
    _check("moe_workspace_views_ec", lib.moe_workspace_views_ec(
        ctypes.byref(cfg), _ptr(ws), *[ctypes.byref(o) for o in outs]))
    return [o.value for o in outs]


def moe_selftest_timeout(ws, limit_us, stream=None):
    _check("moe_selftest_timeout", lib.moe_selftest_timeout(_ptr(ws), int(limit_us),
                                                            _stream(stream)))


def router_backward_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _check("moe_router_backward_workspace_size",
           lib.moe_router_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def router_backward_workspace(cfg: MoeConfig, device="cuda"):
    """A zeroed device workspace for moe_router_backward (torch allocation)."""
    import torch
    return torch.zeros(router_backward_workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_router_backward(cfg, x, w_gate, logits, topk_idx, d_topk_w, f, alpha, beta, d_logits,
                        d_w_gate, d_x, ws, stream=None):
    _check("moe_router_backward", lib.moe_router_backward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(logits), _ptr(topk_idx), _ptr(d_topk_w),
        _ptr(f), float(alpha), float(beta), _ptr(d_logits), _ptr(d_w_gate), _ptr(d_x), _ptr(ws),
        _stream(stream)))


def moe_bias_update(cfg, f, bias, gamma, stream=None):
    _check("moe_bias_update", lib.moe_bias_update(ctypes.byref(cfg), _ptr(f), _ptr(bias),
                                                  float(gamma), _stream(stream)))


def moe_quantize_fp8(src, dst, scale, stream=None):
    """Per-row E4M3 quantisation of a bf16 tensor (leading dimensions flattened into rows):
    dst uint8 of the same shape receives the codes, scale float32 [rows] the row scales."""
    cols = src.shape[-1]
    rows = src.numel() // cols
    _check("moe_quantize_fp8", lib.moe_quantize_fp8(rows, cols, _ptr(src), _ptr(dst), _ptr(scale),
                                                    _stream(stream)))


def quantize_fp8(src, stream=None):
    """Codes (uint8, shape of src) and row scales (float32 [rows]) of a bf16 device tensor."""
    import torch
    dst = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scale = torch.empty(src.numel() // src.shape[-1], dtype=torch.float32, device=src.device)
    moe_quantize_fp8(src, dst, scale, stream)
    return dst, scale


def fp8_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _check("moe_fp8_workspace_size",
           lib.moe_fp8_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def fp8_workspace(cfg: MoeConfig, device="cuda"):
    """A zeroed device workspace for moe_forward_fp8 (torch allocation)."""
    import torch
    return torch.zeros(fp8_workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_forward_fp8(cfg, x, w_gate, bias, w13_q, w13_s, w2_q, w2_s, ws13_q, ws13_s, ws2_q, ws2_s,
                    out, topk_idx=None, topk_w=None, f=None, P=None, l_balance=None, z_loss=None,
                    n_dropped=None, ws=None, stream=None):
    _check("moe_forward_fp8", lib.moe_forward_fp8(
        ctypes.byref(cfg), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(w13_q), _ptr(w13_s),
        _ptr(w2_q), _ptr(w2_s), _ptr(ws13_q), _ptr(ws13_s), _ptr(ws2_q), _ptr(ws2_s), _ptr(out),
        _ptr(topk_idx), _ptr(topk_w), _ptr(f), _ptr(P), _ptr(l_balance), _ptr(z_loss),
        _ptr(n_dropped), _ptr(ws), _stream(stream)))
