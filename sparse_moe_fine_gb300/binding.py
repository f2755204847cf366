"""Thin Python binding of libusaf.so (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls, without the ``usaf_`` prefix.
Tensors are PyTorch CUDA tensors; the binding passes their device pointers and the current CUDA
stream. PyTorch allocates memory and owns streams; every step of the computation runs in the
library's kernels. If the library is missing the binding raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

from . import build as _build

_LIB = None

F32, BF16 = 0, 1
ROW_ALIGN = 16
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "CUDA error",
          5: "timeout"}
DEV_NONFINITE, DEV_SELECT_EXACT_PATH, DEV_TIMEOUT, DEV_BAD_INDEX = 1, 2, 4, 8
DEV_SKIP_MASK = DEV_NONFINITE | DEV_TIMEOUT | DEV_BAD_INDEX


class UsafError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("E", ctypes.c_int64),
                ("k", ctypes.c_int64), ("I", ctypes.c_int64)]


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


class _Routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("topk_idx", "topk_w", "expert_count",
                                               "expert_offset", "perm_tok", "perm_slot",
                                               "slot_row")]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_D = ctypes.c_double
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGS = {
    "usaf_abi_version": (ctypes.c_int, []),
    "usaf_status_string": (ctypes.c_char_p, [_INT]),
    "usaf_routed_rows_capacity": (_I64, [_P]),
    "usaf_route_topk_workspace_size": (_SZ, [_P]),
    "usaf_route_topk": (_INT, [_P, _P, _INT, _P, _P, _P, _INT, _P, _P, _P, _SZ, _P]),
    "usaf_route_topk_noalloc": (_INT, [_P, _P, _INT, _P, _P, _P, _INT, _P, _P, _P]),
    "usaf_moe_fwd_workspace_size": (_SZ, [_P, _INT]),
    "usaf_moe_fwd": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "usaf_moe_fwd_wait": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                 _P]),
    "usaf_moe_bwd_workspace_size": (_SZ, [_P, _INT, _I64]),
    "usaf_moe_bwd_sparse": (_INT, [_P, _INT, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "usaf_sparse_adam_step": (_INT, [_I64, _P, _P, _P, _P, _P, _P, _I64, _P, _INT, _D, _D, _D, _D,
                                     _I64, _INT, _P, _P]),
    "usaf_importance_select_workspace_size": (_SZ, [_I64, _I64]),
    "usaf_importance_select": (_INT, [_P, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "usaf_rigl_swap_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "usaf_trace_enable": (_INT, [_INT]),
    "usaf_launch_count": (_I64, []),
    "usaf_trace_summary": (_INT, [_P, _INT]),
    "usaf_rigl_swap": (_INT, [_P, _I64, _P, _I64, _I64, _P, _P, _P, _P, _I64, _P, _INT, _P, _P, _P,
                              _P, _P, _P, _P, _SZ, _P]),
    "usaf_moe_fwd_wait2": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _SZ, _P]),
    "usaf_moe_fwd_stage": (_INT, [_P, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _INT, _P, _P, _SZ,
                                  _P]),
    "usaf_scan_nonfinite": (_INT, [_P, _I64, _P, _P]),
    "usaf_select_and_swap_workspace_size": (_SZ, [_I64, _I64, _I64, _I64]),
    "usaf_select_and_swap": (_INT, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, _P, _P, _I64, _P,
                                    _INT, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "usaf_moe_bwd_sparse_accumulate": (_INT, [_P, _INT, _INT, _P, _P, _P, _P, _P, _P, _P, _P,
                                              _P, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _SZ,
                                              _P]),
    "usaf_moe_bwd_dense": (_INT, [_P, _INT, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _INT, _P, _P, _P, _P, _P, _SZ, _P]),
    "usaf_validate_active": (_INT, [_P, _I64, _I64, _P, _P]),
    "usaf_shard_key_histogram": (_INT, [_P, _I64, _P, ctypes.c_uint32, _INT, _INT, _P, _P]),
    "usaf_shard_emit_workspace_size": (_SZ, [_I64, _I64]),
    "usaf_shard_emit": (_INT, [_P, _I64, _P, ctypes.c_uint32, _I64, _I64, _I64, _P, _P, _P, _SZ,
                               _P]),
    "usaf_active_bitmap": (_INT, [_P, _I64, _I64, _I64, _P, _P]),
    "usaf_rigl_apply_workspace_size": (_SZ, [_I64, _I64]),
    "usaf_rigl_apply": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I64, _P, _INT, _P, _P,
                               _P, _P, _P, _P, _P, _SZ, _P]),
    "usaf_reselect_carry_workspace_size": (_SZ, []),
    "usaf_reselect_carry": (_INT, [_P, _I64, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _INT, _P,
                                   _P, _P, _P, _P, _P, _SZ, _P]),
    "usaf_masked_plan_size": (_SZ, [_P]),
    "usaf_masked_plan_build": (_INT, [_P, _P, _I64, _D, _P, _SZ, _P]),
    "usaf_moe_bwd_sparse_planned": (_INT, [_P, _INT, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _P, _P, _I64, _P, _P, _P, _P, _INT, _P, _I64, _P, _P,
                                           _SZ, _P]),
    "usaf_moe_wgrad_dense": (_INT, [_P, _INT, _P, _P, _P, _P, _INT, _P, _P, _SZ, _P]),
    "usaf_moe_bwd_dlogit_offset": (_I64, [_P, _INT, _I64]),
    "usaf_diag_bounded_wait": (_INT, [_I64, _P, _P]),
    "usaf_reselect_full_workspace_size": (_SZ, [_I64, _I64]),
    "usaf_reselect_full": (_INT, [_P, _I64, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _INT, _P,
                                  _P, _P, _P, _P, _P, _P, _SZ, _P]),
}


def header_symbols() -> list:
    """Names of the functions include/usaf.h declares."""
    text = open(os.path.join(_build.ROOT, "include", "usaf.h")).read()
    return sorted(set(re.findall(r"\b(usaf_[a-z0-9_]+)\s*\(", text)))


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load libusaf.so (building it first if it is absent)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            _build.build()
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(name: str, code: int) -> None:
    if code != 0:
        raise UsafError(name, code)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def shape(T, H, E, k, I) -> Shape:
    return Shape(int(T), int(H), int(E), int(k), int(I))


def routed_rows_capacity(s: Shape) -> int:
    return int(lib().usaf_routed_rows_capacity(ctypes.byref(s)))


@dataclass
class Routing:
    """Device routing tables of one layer call (see usaf_routing in include/usaf.h)."""
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    expert_count: torch.Tensor
    expert_offset: torch.Tensor
    perm_tok: torch.Tensor
    perm_slot: torch.Tensor
    slot_row: torch.Tensor

    @staticmethod
    def empty(s: Shape, device="cuda") -> "Routing":
        R = s.T * s.k
        cap = routed_rows_capacity(s)
        i32 = dict(dtype=torch.int32, device=device)
        return Routing(torch.empty(R, **i32), torch.empty(R, dtype=torch.float32, device=device),
                       torch.empty(s.E, **i32), torch.empty(s.E + 1, **i32),
                       torch.empty(cap, **i32), torch.empty(cap, **i32), torch.empty(R, **i32))

    def c(self) -> _Routing:
        return _Routing(*[_ptr(getattr(self, f)) for f, _ in _Routing._fields_])


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def route_topk_workspace_size(s: Shape) -> int:
    return int(lib().usaf_route_topk_workspace_size(ctypes.byref(s)))


def route_topk(s: Shape, x, w_router, rt: Routing, logits_in=None, logits_out=None, renorm=1,
               dev_status=None, ws=None, stream=None):
    dev = rt.topk_idx.device
    if ws is None:
        ws = _ws(route_topk_workspace_size(s), dev)
    xdt = _dt(x) if x is not None else F32
    r = rt.c()
    _check("usaf_route_topk", lib().usaf_route_topk(
        ctypes.byref(s), _ptr(x), xdt, _ptr(w_router), _ptr(logits_in), _ptr(logits_out),
        int(renorm), ctypes.byref(r), _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def route_topk_noalloc(s: Shape, x, w_router, rt: Routing, logits_in=None, logits_out=None,
                       renorm=1, dev_status=None, stream=None):
    """usaf_route_topk_noalloc: no workspace argument; scratch is the library's fixed array."""
    xdt = _dt(x) if x is not None else F32
    r = rt.c()
    _check("usaf_route_topk_noalloc", lib().usaf_route_topk_noalloc(
        ctypes.byref(s), _ptr(x), xdt, _ptr(w_router), _ptr(logits_in), _ptr(logits_out),
        int(renorm), ctypes.byref(r), _ptr(dev_status), _stream(stream)))


def moe_fwd_workspace_size(s: Shape, dt: int) -> int:
    return int(lib().usaf_moe_fwd_workspace_size(ctypes.byref(s), dt))


def moe_fwd(s: Shape, x, w_gate_up, w_down, rt: Routing, x_perm, h, wa, y, ws=None, stream=None,
            weights_ready=None, dev_status=None, down_ready=None):
    """weights_ready: a recorded torch.cuda.Event that the reads of the expert weights wait for
    (the token gather before them does not); with down_ready, weights_ready is waited for before
    the gate_up GEMM and down_ready before the down GEMM (usaf_moe_fwd_wait2)."""
    dt = _dt(x)
    if ws is None:
        ws = _ws(moe_fwd_workspace_size(s, dt), x.device)
    r = rt.c()
    ev = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    if down_ready is None:
        _check("usaf_moe_fwd_wait", lib().usaf_moe_fwd_wait(
            ctypes.byref(s), dt, _ptr(x), _ptr(w_gate_up), _ptr(w_down), ctypes.byref(r),
            _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(y), ev(weights_ready), _ptr(dev_status),
            _ptr(ws), ws.numel(), _stream(stream)))
    else:
        _check("usaf_moe_fwd_wait2", lib().usaf_moe_fwd_wait2(
            ctypes.byref(s), dt, _ptr(x), _ptr(w_gate_up), _ptr(w_down), ctypes.byref(r),
            _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(y), ev(weights_ready), ev(down_ready),
            _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


FWD_GATHER, FWD_GATE_UP, FWD_DOWN = 1, 2, 4


def moe_fwd_stage(s: Shape, x, w_gate_up, w_down, rt: Routing, x_perm, h, wa, y, stages, ws,
                  stream=None, dev_status=None):
    """usaf_moe_fwd_stage: the forward's stages in the bit set `stages` (FWD_GATHER,
    FWD_GATE_UP, FWD_DOWN), in order, on the workspace the earlier stages used."""
    r = rt.c()
    _check("usaf_moe_fwd_stage", lib().usaf_moe_fwd_stage(
        ctypes.byref(s), _dt(x), _ptr(x), _ptr(w_gate_up), _ptr(w_down), ctypes.byref(r),
        _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(y), int(stages), _ptr(dev_status), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_bwd_workspace_size(s: Shape, dt: int, K: int) -> int:
    return int(lib().usaf_moe_bwd_workspace_size(ctypes.byref(s), dt, int(K)))


def moe_bwd_dlogit_offset(s: Shape, dt: int, K: int) -> int:
    """Byte offset in the backward workspace of dlogit at the selected experts ([T*k] fp32)."""
    return int(lib().usaf_moe_bwd_dlogit_offset(ctypes.byref(s), dt, int(K)))


def moe_bwd_sparse(s: Shape, x, w_router, w_gate_up, w_down, rt: Routing, x_perm, h, wa, dy,
                   act_idx, g_act, g_router, dx=None, dw_slot=None, logits=None, renorm=1,
                   dev_status=None, ws=None, stream=None):
    dt = _dt(x)
    K = 0 if act_idx is None else act_idx.numel()
    if ws is None:
        ws = _ws(moe_bwd_workspace_size(s, dt, K), x.device)
    r = rt.c()
    _check("usaf_moe_bwd_sparse", lib().usaf_moe_bwd_sparse(
        ctypes.byref(s), dt, int(renorm), _ptr(x), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down),
        ctypes.byref(r), _ptr(logits), _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(dy), _ptr(act_idx),
        K, _ptr(g_act), _ptr(g_router), _ptr(dx), _ptr(dw_slot), _ptr(dev_status), _ptr(ws),
        ws.numel(), _stream(stream)))


def masked_plan_size(s: Shape) -> int:
    return int(lib().usaf_masked_plan_size(ctypes.byref(s)))


def masked_plan_build(s: Shape, act_idx, dense_density, plan, stream=None):
    """usaf_masked_plan_build; after the stream has run it, masked_plan_count(plan) reads the
    number of listed experts."""
    K = 0 if act_idx is None else act_idx.numel()
    _check("usaf_masked_plan_build", lib().usaf_masked_plan_build(
        ctypes.byref(s), _ptr(act_idx), K, float(dense_density), _ptr(plan), plan.numel(),
        _stream(stream)))


def masked_plan_count(plan) -> int:
    """The plan's first 8 bytes: the number of experts it lists (reads device memory)."""
    return int(plan[:8].view(torch.int64).item())


def moe_bwd_sparse_planned(s: Shape, x, w_router, w_gate_up, w_down, rt: Routing, x_perm, h, wa,
                           dy, act_idx, g_act, g_router, plan=None, n_dense=0, accumulate=0,
                           dx=None, dw_slot=None, logits=None, renorm=1, dev_status=None,
                           ws=None, stream=None):
    dt = _dt(x)
    K = 0 if act_idx is None else act_idx.numel()
    if ws is None:
        ws = _ws(moe_bwd_workspace_size(s, dt, K), x.device)
    r = rt.c()
    _check("usaf_moe_bwd_sparse_planned", lib().usaf_moe_bwd_sparse_planned(
        ctypes.byref(s), dt, int(renorm), _ptr(x), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down),
        ctypes.byref(r), _ptr(logits), _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(dy), _ptr(act_idx),
        K, _ptr(g_act), _ptr(g_router), _ptr(dx), _ptr(dw_slot), int(accumulate), _ptr(plan),
        int(n_dense), _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def moe_bwd_sparse_accumulate(s: Shape, x, w_router, w_gate_up, w_down, rt: Routing, x_perm,
                              h, wa, dy, act_idx, g_act, g_router, dx=None, dw_slot=None,
                              logits=None, renorm=1, dev_status=None, ws=None, stream=None):
    """moe_bwd_sparse that adds this micro-batch's g_act and g_router to the buffers."""
    dt = _dt(x)
    K = 0 if act_idx is None else act_idx.numel()
    if ws is None:
        ws = _ws(moe_bwd_workspace_size(s, dt, K), x.device)
    r = rt.c()
    _check("usaf_moe_bwd_sparse_accumulate", lib().usaf_moe_bwd_sparse_accumulate(
        ctypes.byref(s), dt, int(renorm), _ptr(x), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down),
        ctypes.byref(r), _ptr(logits), _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(dy), _ptr(act_idx),
        K, _ptr(g_act), _ptr(g_router), _ptr(dx), _ptr(dw_slot), _ptr(dev_status), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_bwd_dense(s: Shape, x, w_router, w_gate_up, w_down, rt: Routing, x_perm, h, wa, dy,
                  g_dense, g_router, accumulate=0, dx=None, dw_slot=None, logits=None, renorm=1,
                  dev_status=None, ws=None, stream=None):
    dt = _dt(x)
    if ws is None:
        ws = _ws(moe_bwd_workspace_size(s, dt, 0), x.device)
    r = rt.c()
    _check("usaf_moe_bwd_dense", lib().usaf_moe_bwd_dense(
        ctypes.byref(s), dt, int(renorm), _ptr(x), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down),
        ctypes.byref(r), _ptr(logits), _ptr(x_perm), _ptr(h), _ptr(wa), _ptr(dy), _ptr(g_dense),
        int(accumulate), _ptr(g_router), _ptr(dx), _ptr(dw_slot), _ptr(dev_status), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_wgrad_dense(s: Shape, rt: Routing, x_perm, wa, g_dense, ws, accumulate=0,
                    dev_status=None, stream=None):
    """usaf_moe_wgrad_dense: the dense expert gradient from the dh and permuted dy that the last
    backward call left in `ws` (that call's workspace)."""
    r = rt.c()
    _check("usaf_moe_wgrad_dense", lib().usaf_moe_wgrad_dense(
        ctypes.byref(s), _dt(x_perm), ctypes.byref(r), _ptr(x_perm), _ptr(wa), _ptr(g_dense),
        int(accumulate), _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def sparse_adam_step(idx, g, p, m, v, w_seg0, n_seg0, w_seg1, lr, beta1, beta2, eps, step,
                     skip_if_nonfinite=0, dev_status=None, stream=None, n=None):
    n = g.numel() if n is None else n
    _check("usaf_sparse_adam_step", lib().usaf_sparse_adam_step(
        int(n), _ptr(idx), _ptr(g), _ptr(p), _ptr(m), _ptr(v), _ptr(w_seg0), int(n_seg0),
        _ptr(w_seg1), _dt(w_seg0), float(lr), float(beta1), float(beta2), float(eps), int(step),
        int(skip_if_nonfinite), _ptr(dev_status), _stream(stream)))


def scan_nonfinite(g, dev_status, stream=None, n=None):
    """usaf_scan_nonfinite: sets DEV_NONFINITE in dev_status when g[:n] holds a NaN or inf."""
    n = g.numel() if n is None else n
    _check("usaf_scan_nonfinite", lib().usaf_scan_nonfinite(_ptr(g), int(n), _ptr(dev_status),
                                                            _stream(stream)))


def importance_select_workspace_size(N: int, K: int) -> int:
    return int(lib().usaf_importance_select_workspace_size(int(N), int(K)))


def importance_select(g, K, out_idx, dev_status=None, ws=None, stream=None):
    N = g.numel()
    if ws is None:
        ws = _ws(importance_select_workspace_size(N, K), g.device)
    _check("usaf_importance_select", lib().usaf_importance_select(
        _ptr(g), N, int(K), _ptr(out_idx), _ptr(dev_status), _ptr(ws), ws.numel(),
        _stream(stream)))


def rigl_swap_workspace_size(N: int, K: int, D: int) -> int:
    return int(lib().usaf_rigl_swap_workspace_size(int(N), int(K), int(D)))


def rigl_swap(g, act_idx, D, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1, new_idx, p_out, m_out,
              v_out, n_swapped, dev_status=None, ws=None, stream=None):
    N, K = g.numel(), act_idx.numel()
    if ws is None:
        ws = _ws(rigl_swap_workspace_size(N, K, D), g.device)
    _check("usaf_rigl_swap", lib().usaf_rigl_swap(
        _ptr(g), N, _ptr(act_idx), K, int(D), _ptr(p_in), _ptr(m_in), _ptr(v_in), _ptr(w_seg0),
        int(n_seg0), _ptr(w_seg1), _dt(w_seg0), _ptr(new_idx), _ptr(p_out), _ptr(m_out),
        _ptr(v_out), _ptr(n_swapped), _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def select_and_swap_workspace_size(N: int, K_sel: int, K: int, D: int) -> int:
    return int(lib().usaf_select_and_swap_workspace_size(int(N), int(K_sel), int(K), int(D)))


def select_and_swap(g, sel_idx, act_idx, D, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1, new_idx,
                    p_out, m_out, v_out, n_swapped, dev_status=None, ws=None, stream=None):
    """usaf_select_and_swap: importance_select into sel_idx (K_sel = its length) and rigl_swap of
    act_idx, from one pass over g."""
    N, K, K_sel = g.numel(), act_idx.numel(), sel_idx.numel()
    if ws is None:
        ws = _ws(select_and_swap_workspace_size(N, K_sel, K, D), g.device)
    _check("usaf_select_and_swap", lib().usaf_select_and_swap(
        _ptr(g), N, K_sel, _ptr(sel_idx), _ptr(act_idx), K, int(D), _ptr(p_in), _ptr(m_in),
        _ptr(v_in), _ptr(w_seg0), int(n_seg0), _ptr(w_seg1), _dt(w_seg0), _ptr(new_idx),
        _ptr(p_out), _ptr(m_out), _ptr(v_out), _ptr(n_swapped), _ptr(dev_status), _ptr(ws),
        ws.numel(), _stream(stream)))


def reselect_full_workspace_size(N: int, K: int) -> int:
    return int(lib().usaf_reselect_full_workspace_size(int(N), int(K)))


def reselect_full(g, K, old_idx, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1, new_idx, p_out, m_out,
                  v_out, n_kept, dev_status=None, ws=None, stream=None):
    N, K_old = g.numel(), old_idx.numel()
    if ws is None:
        ws = _ws(reselect_full_workspace_size(N, K), g.device)
    _check("usaf_reselect_full", lib().usaf_reselect_full(
        _ptr(g), N, int(K), _ptr(old_idx), K_old, _ptr(p_in), _ptr(m_in), _ptr(v_in),
        _ptr(w_seg0), int(n_seg0), _ptr(w_seg1), _dt(w_seg0), _ptr(new_idx), _ptr(p_out),
        _ptr(m_out), _ptr(v_out), _ptr(n_kept), _ptr(dev_status), _ptr(ws), ws.numel(),
        _stream(stream)))


def validate_active(idx, N, dev_status, stream=None):
    """usaf_validate_active: sets DEV_BAD_INDEX in dev_status unless idx is strictly ascending in
    [0, N)."""
    K = 0 if idx is None else idx.numel()
    _check("usaf_validate_active", lib().usaf_validate_active(
        _ptr(idx), K, int(N), _ptr(dev_status), _stream(stream)))


def diag_bounded_wait(limit_cycles, dev_status, stream=None):
    """usaf_diag_bounded_wait: one CTA whose bounded mbarrier wait runs out after limit_cycles."""
    _check("usaf_diag_bounded_wait", lib().usaf_diag_bounded_wait(
        int(limit_cycles), _ptr(dev_status), _stream(stream)))


def shard_key_histogram(g, excl, prefix, shift, bits, hist, stream=None):
    """hist [2^bits] uint64 (int64 tensor) += digit counts of the part's keys (usaf.h)."""
    _check("usaf_shard_key_histogram", lib().usaf_shard_key_histogram(
        _ptr(g), g.numel(), _ptr(excl), int(prefix) & 0xFFFFFFFF, int(shift), int(bits),
        _ptr(hist), _stream(stream)))


def shard_emit(g, excl, tau, take_eq, count, base, out, dev_status=None, ws=None, stream=None):
    n = g.numel()
    if ws is None:
        ws = _ws(lib().usaf_shard_emit_workspace_size(n, int(count)), g.device)
    _check("usaf_shard_emit", lib().usaf_shard_emit(
        _ptr(g), n, _ptr(excl), int(tau) & 0xFFFFFFFF, int(take_eq), int(count), int(base),
        _ptr(out), _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def active_bitmap(idx, lo, n, bitmap, stream=None):
    K = 0 if idx is None else idx.numel()
    _check("usaf_active_bitmap", lib().usaf_active_bitmap(
        _ptr(idx), K, int(lo), int(n), _ptr(bitmap), _stream(stream)))


def _n_entries(n_seg0, w_seg1):
    return int(n_seg0) + (0 if w_seg1 is None else w_seg1.numel())


def rigl_apply(act_idx, D, grown, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1, new_idx, p_out,
               m_out, v_out, n_swapped, dev_status=None, ws=None, stream=None):
    """usaf_rigl_apply: RigL's drop and merge with the grow set given (chosen over ranks)."""
    K = act_idx.numel()
    if ws is None:
        ws = _ws(lib().usaf_rigl_apply_workspace_size(K, int(D)), act_idx.device)
    _check("usaf_rigl_apply", lib().usaf_rigl_apply(
        _ptr(act_idx), K, _n_entries(n_seg0, w_seg1), int(D), _ptr(grown), _ptr(p_in), _ptr(m_in), _ptr(v_in), _ptr(w_seg0),
        int(n_seg0), _ptr(w_seg1), _dt(w_seg0), _ptr(new_idx), _ptr(p_out), _ptr(m_out),
        _ptr(v_out), _ptr(n_swapped), _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def reselect_carry(new_idx, old_idx, p_in, m_in, v_in, w_seg0, n_seg0, w_seg1, p_out, m_out,
                   v_out, n_kept, dev_status=None, ws=None, stream=None):
    """usaf_reselect_carry: the state of a full reselection for a new set chosen over ranks."""
    if ws is None:
        ws = _ws(lib().usaf_reselect_carry_workspace_size(), new_idx.device)
    _check("usaf_reselect_carry", lib().usaf_reselect_carry(
        _ptr(new_idx), new_idx.numel(), _n_entries(n_seg0, w_seg1), _ptr(old_idx),
        old_idx.numel(), _ptr(p_in), _ptr(m_in), _ptr(v_in), _ptr(w_seg0), int(n_seg0),
        _ptr(w_seg1), _dt(w_seg0), _ptr(p_out), _ptr(m_out), _ptr(v_out), _ptr(n_kept),
        _ptr(dev_status), _ptr(ws), ws.numel(), _stream(stream)))


def trace_enable(on: bool) -> None:
    _check("usaf_trace_enable", lib().usaf_trace_enable(1 if on else 0))


def trace_summary() -> list:
    """[(kernel name, launches, total ms)] of the launches recorded since trace_enable(True)."""
    L = lib()
    n = L.usaf_trace_summary(None, 0)
    if n < 0:
        raise UsafError("usaf_trace_summary", 4)
    arr = (TraceEntry * max(n, 1))()
    n = L.usaf_trace_summary(arr, n)
    return [(arr[i].name.decode(), int(arr[i].launches), float(arr[i].total_ms)) for i in range(n)]


def launch_count() -> int:
    """Kernel launches the library has issued since it was loaded."""
    return int(lib().usaf_launch_count())
