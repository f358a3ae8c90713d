"""Thin Python binding of libep_gb300.so (the C ABI in include/ep.h).

Functions carry the C names and only marshal arguments: they check that each
tensor is a contiguous CUDA tensor of the right dtype and shape, pass its
device address and the current CUDA stream, and raise :class:`EpError` on a
non-OK status.  Every step runs in the library's sm_103a kernels; there is no
CPU path.  ``alloc_*`` helpers allocate output tensors with torch.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = -1
EP_ERR_CUDA = -2
EP_ERR_CAPACITY = -3
EP_ERR_TIMEOUT = -4
EP_ERR_INCONSISTENT = -5
EP_ERR_INPUT = -6

EP_DEV_CAPACITY = 0x1
EP_DEV_TIMEOUT = 0x2
EP_DEV_INCONSISTENT = 0x4
EP_DEV_INPUT = 0x8

NODE_SIZE = 8

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class EpShape(ctypes.Structure):
    """Mirror of ep_shape_t."""

    _fields_ = [("num_ranks", _i32), ("num_tokens", _i32), ("num_topk", _i32),
                ("num_experts", _i32), ("hidden", _i32), ("num_channels", _i32),
                ("expert_alignment", _i32)]

    @classmethod
    def make(cls, R, T, K, E, H, C, expert_alignment=1) -> "EpShape":
        return cls(R, T, K, E, H, C, expert_alignment)

    @property
    def N(self) -> int:
        return 1 if self.num_ranks <= NODE_SIZE else self.num_ranks // NODE_SIZE

    @property
    def E_loc(self) -> int:
        return self.num_experts // self.num_ranks


class EpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {ep_status_string(status)} ({status})")


_SIGS = {
    "ep_status_string": (ctypes.c_char_p, [_i32]),
    "ep_check_shape": (_i32, [ctypes.POINTER(EpShape)]),
    "ep_num_nodes": (_i32, [ctypes.POINTER(EpShape)]),
    "ep_notify_workspace_bytes": (_sz, [ctypes.POINTER(EpShape)]),
    "ep_get_dispatch_layout": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 6 + [_vp]),
    "ep_notify_dispatch": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 16 + [_sz, _vp, _vp, _vp]),
    "ep_dispatch": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 5 + [_i64] + [_vp] * 6 + [_vp]),
    "ep_dispatch_fp8": (_i32, [ctypes.POINTER(EpShape), _vp, _vp, _i32] + [_vp] * 4 + [_i64] +
                        [_vp] * 7 + [_vp]),
    "ep_combine": (_i32, [ctypes.POINTER(EpShape), _vp, _vp, _i64] + [_vp] * 5 + [_vp]),
    "ep_layout_notify": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 16 + [_vp, _sz, _vp, _vp, _vp]),
    "ep_layout_notify_fused": (_i32, [ctypes.POINTER(EpShape)]),
    "ep_layout_notify_workspace_bytes": (_sz, [ctypes.POINTER(EpShape)]),
    "ep_debug_layout_notify_tiled": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 16 +
                                     [_vp, _sz, _vp, _vp, _i32, _i32, _i32, _vp]),
    "ep_layout_notify_dispatch": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 18 + [_vp, _sz, _i64] + [_vp] * 7 +
                                  [_vp]),
    "ep_debug_layout_notify_dispatch_stall": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 18 + [_vp, _sz, _i64] +
                                              [_vp] * 6 + [_i32, _i32, _vp]),
    "ep_notify_dispatch_noalloc": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 15 + [_vp, _vp, _vp]),
    "ep_ll_layout": (_i32, [ctypes.POINTER(EpShape), _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "ep_ll_dispatch": (_i32, [ctypes.POINTER(EpShape), _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "ep_ll_combine": (_i32, [ctypes.POINTER(EpShape), _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ep_sync_status": (_i32, [_vp, _vp]),
    "ep_debug_notify_dispatch_stall": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 16 +
                                       [_sz, _vp, _i32, _i32, _vp]),
    "ep_debug_dispatch_stall": (_i32, [ctypes.POINTER(EpShape)] + [_vp] * 5 + [_i64] + [_vp] * 6 +
                                [_i32, _i32, _vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libep_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c \"import "
                               "__graft_entry__ as g; g.build()\"` (needs nvcc)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


# --------------------------------------------------------------------------- helpers
def _stream(stream) -> _vp:
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _t(t: torch.Tensor | None, dtype, shape, name: str, nullable=False) -> _vp:
    if t is None:
        if nullable:
            return _vp(None)
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return _vp(t.data_ptr())


def _rows(t: torch.Tensor, name: str) -> int:
    if t.dim() < 1:
        raise ValueError(f"{name} must have a row axis")
    return t.shape[0]


def _check(fn: str, rc: int) -> None:
    if rc != EP_OK:
        raise EpError(fn, rc)


# --------------------------------------------------------------------------- C names
def ep_status_string(status: int) -> str:
    return lib().ep_status_string(status).decode()


def ep_check_shape(shape: EpShape) -> int:
    return lib().ep_check_shape(ctypes.byref(shape))


def ep_num_nodes(shape: EpShape) -> int:
    return lib().ep_num_nodes(ctypes.byref(shape))


def ep_notify_workspace_bytes(shape: EpShape) -> int:
    return int(lib().ep_notify_workspace_bytes(ctypes.byref(shape)))


def ep_get_dispatch_layout(shape: EpShape, topk_idx, num_tokens_per_rank, num_tokens_per_rdma_rank,
                           num_tokens_per_expert, is_token_in_rank, status, stream=None) -> None:
    R, T, K, E, N = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.num_experts, shape.N
    rc = lib().ep_get_dispatch_layout(
        ctypes.byref(shape), _t(topk_idx, torch.int64, (R, T, K), "topk_idx"),
        _t(num_tokens_per_rank, torch.int32, (R, R), "num_tokens_per_rank"),
        _t(num_tokens_per_rdma_rank, torch.int32, (R, N), "num_tokens_per_rdma_rank"),
        _t(num_tokens_per_expert, torch.int32, (R, E), "num_tokens_per_expert"),
        _t(is_token_in_rank, torch.uint8, (R, T, R), "is_token_in_rank"),
        _t(status, torch.int32, (1,), "status"), _stream(stream))
    _check("ep_get_dispatch_layout", rc)


_NOTIFY_OUT = ("rank_prefix_matrix", "gbl_channel_prefix_matrix", "rdma_channel_prefix_matrix",
               "recv_gbl_rank_prefix_sum", "recv_rdma_rank_prefix_sum", "recv_channel_offset",
               "num_recv_tokens", "num_rdma_recv_tokens", "num_recv_tokens_per_expert", "recv_base",
               "send_pos")


def notify_shapes(shape: EpShape) -> dict:
    R, T, C, N, El = shape.num_ranks, shape.num_tokens, shape.num_channels, shape.N, shape.E_loc
    return dict(
        rank_prefix_matrix=((R, R), torch.int32),
        gbl_channel_prefix_matrix=((R, R, C), torch.int32),
        rdma_channel_prefix_matrix=((R, N, C), torch.int32),
        recv_gbl_rank_prefix_sum=((R, R), torch.int32),
        recv_rdma_rank_prefix_sum=((R, N), torch.int32),
        recv_channel_offset=((R, R, C), torch.int32),
        num_recv_tokens=((R,), torch.int32),
        num_rdma_recv_tokens=((R,), torch.int32),
        num_recv_tokens_per_expert=((R, El), torch.int32),
        recv_base=((R + 1,), torch.int64),
        send_pos=((R, T, R), torch.int32),
    )


def _notify_args(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                 num_tokens_per_expert, outs: dict):
    R, T, E, N = shape.num_ranks, shape.num_tokens, shape.num_experts, shape.N
    shapes = notify_shapes(shape)
    args = [_t(is_token_in_rank, torch.uint8, (R, T, R), "is_token_in_rank"),
            _t(num_tokens_per_rank, torch.int32, (R, R), "num_tokens_per_rank"),
            _t(num_tokens_per_rdma_rank, torch.int32, (R, N), "num_tokens_per_rdma_rank"),
            _t(num_tokens_per_expert, torch.int32, (R, E), "num_tokens_per_expert")]
    for k in _NOTIFY_OUT:
        shp, dt = shapes[k]
        args.append(_t(outs[k], dt, shp, k))
    return args


def ep_notify_dispatch(shape: EpShape, is_token_in_rank, num_tokens_per_rank,
                       num_tokens_per_rdma_rank, num_tokens_per_expert, outs: dict, workspace,
                       status, host_num_recv_tokens=None, stream=None) -> None:
    """``outs`` maps each notify output name (see :func:`notify_shapes`) to its tensor.
    ``host_num_recv_tokens`` may be a pinned, host-mapped int32 tensor of R+1."""
    args = _notify_args(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                        num_tokens_per_expert, outs)
    need = ep_notify_workspace_bytes(shape)
    if workspace is None or not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    host = _vp(None)
    if host_num_recv_tokens is not None:
        if host_num_recv_tokens.dtype != torch.int32 or host_num_recv_tokens.numel() < shape.num_ranks + 1:
            raise ValueError("host_num_recv_tokens must be int32 with R+1 elements")
        host = _vp(host_num_recv_tokens.data_ptr())
    rc = lib().ep_notify_dispatch(ctypes.byref(shape), *args, _vp(workspace.data_ptr()),
                                  _sz(workspace.numel() * workspace.element_size()),
                                  _t(status, torch.int32, (1,), "status"), host, _stream(stream))
    _check("ep_notify_dispatch", rc)


def ep_layout_notify_fused(shape: EpShape) -> int:
    """Which kernel :func:`ep_layout_notify` runs for ``shape`` on the current
    device: 1 = the cluster form, 2 = the tiled form (both one launch)."""
    return int(lib().ep_layout_notify_fused(ctypes.byref(shape)))


def ep_layout_notify_workspace_bytes(shape: EpShape) -> int:
    return int(lib().ep_layout_notify_workspace_bytes(ctypes.byref(shape)))


def _layout_notify_args(shape, topk_idx, layout: dict, outs: dict):
    R, T, K, E, N = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.num_experts, shape.N
    shapes = notify_shapes(shape)
    args = [_t(topk_idx, torch.int64, (R, T, K), "topk_idx"),
            _t(layout["num_tokens_per_rank"], torch.int32, (R, R), "num_tokens_per_rank"),
            _t(layout["num_tokens_per_rdma_rank"], torch.int32, (R, N), "num_tokens_per_rdma_rank"),
            _t(layout["num_tokens_per_expert"], torch.int32, (R, E), "num_tokens_per_expert"),
            _t(layout["is_token_in_rank"], torch.uint8, (R, T, R), "is_token_in_rank")]
    for k in _NOTIFY_OUT:
        shp, dt = shapes[k]
        args.append(_t(outs[k], dt, shp, k))
    return args


def _host_counts(shape, host_num_recv_tokens) -> _vp:
    if host_num_recv_tokens is None:
        return _vp(None)
    if host_num_recv_tokens.dtype != torch.int32 or host_num_recv_tokens.numel() < shape.num_ranks + 1:
        raise ValueError("host_num_recv_tokens must be int32 with R+1 elements")
    return _vp(host_num_recv_tokens.data_ptr())


def _workspace(workspace, need: int, name="workspace"):
    if workspace is None or not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"{name} must be a CUDA tensor of at least {need} bytes")
    return _vp(workspace.data_ptr()), _sz(workspace.numel() * workspace.element_size())


def ep_layout_notify(shape: EpShape, topk_idx, layout: dict, outs: dict, workspace, status,
                     host_num_recv_tokens=None, stream=None) -> None:
    """Layout and notify in one call.  ``layout`` holds the four layout outputs
    (see :func:`alloc_layout`), ``outs`` the notify outputs (see
    :func:`notify_shapes`); ``workspace`` from :func:`alloc_layout_notify_workspace`."""
    args = _layout_notify_args(shape, topk_idx, layout, outs)
    ws, nws = _workspace(workspace, ep_layout_notify_workspace_bytes(shape))
    rc = lib().ep_layout_notify(ctypes.byref(shape), *args, ws, nws, _t(status, torch.int32, (1,), "status"),
                                _host_counts(shape, host_num_recv_tokens), _stream(stream))
    _check("ep_layout_notify", rc)


def ep_debug_layout_notify_tiled(shape: EpShape, topk_idx, layout: dict, outs: dict, workspace, status,
                                 tile_tokens: int = 0, stall_tile: int = -1, wait_limit_us: int = 1000000,
                                 host_num_recv_tokens=None, stream=None) -> None:
    """Testing hook: :func:`ep_layout_notify` forced onto the tiled form with
    ``tile_tokens`` tokens per tile (0: default) and optionally one tile
    withholding its lookback words."""
    args = _layout_notify_args(shape, topk_idx, layout, outs)
    ws, nws = _workspace(workspace, 0)
    rc = lib().ep_debug_layout_notify_tiled(
        ctypes.byref(shape), *args, ws, nws, _t(status, torch.int32, (1,), "status"),
        _host_counts(shape, host_num_recv_tokens), _i32(tile_tokens), _i32(stall_tile), _i32(wait_limit_us),
        _stream(stream))
    _check("ep_debug_layout_notify_tiled", rc)


def ep_notify_dispatch_noalloc(shape: EpShape, is_token_in_rank, num_tokens_per_rank,
                               num_tokens_per_rdma_rank, num_tokens_per_expert, outs: dict, status,
                               host_num_recv_tokens=None, stream=None) -> None:
    """ep_notify_dispatch using the library's fixed 1 MiB device scratch instead of a
    caller workspace, for callers that cannot allocate device memory.  Calls share
    that scratch, so calls that overlap on the GPU race; ``outs`` needs no
    "workspace" entry."""
    args = _notify_args(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                        num_tokens_per_expert, outs)
    host = _vp(None)
    if host_num_recv_tokens is not None:
        if host_num_recv_tokens.dtype != torch.int32 or host_num_recv_tokens.numel() < shape.num_ranks + 1:
            raise ValueError("host_num_recv_tokens must be int32 with R+1 elements")
        host = _vp(host_num_recv_tokens.data_ptr())
    rc = lib().ep_notify_dispatch_noalloc(ctypes.byref(shape), *args,
                                          _t(status, torch.int32, (1,), "status"), host, _stream(stream))
    _check("ep_notify_dispatch_noalloc", rc)


def ep_debug_notify_dispatch_stall(shape: EpShape, is_token_in_rank, num_tokens_per_rank,
                                   num_tokens_per_rdma_rank, num_tokens_per_expert, outs: dict,
                                   workspace, status, stall_block: int, wait_limit_us: int,
                                   stream=None) -> None:
    args = _notify_args(shape, is_token_in_rank, num_tokens_per_rank, num_tokens_per_rdma_rank,
                        num_tokens_per_expert, outs)
    rc = lib().ep_debug_notify_dispatch_stall(
        ctypes.byref(shape), *args, _vp(workspace.data_ptr()),
        _sz(workspace.numel() * workspace.element_size()), _t(status, torch.int32, (1,), "status"),
        _i32(stall_block), _i32(wait_limit_us), _stream(stream))
    _check("ep_debug_notify_dispatch_stall", rc)


def _sched(sched):
    return _t(sched, torch.int64, (1,), "sched", nullable=True)


def _lnd_args(shape, x, topk_idx, topk_w, layout, outs, workspace, disp, sched):
    R, T, K, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.hidden
    ln = _layout_notify_args(shape, topk_idx, layout, outs)
    cap = _rows(disp["recv_x"], "recv_x")
    ws, nws = _workspace(workspace, ep_layout_notify_workspace_bytes(shape))
    return ([ln[0], _t(topk_w, torch.float32, (R, T, K), "topk_w", nullable=True),
             _t(x, torch.bfloat16, (R, T, H), "x")] + ln[1:] +
            [ws, nws, _i64(cap), _t(disp["recv_x"], torch.bfloat16, (cap, H), "recv_x"),
             _t(disp.get("recv_topk_idx"), torch.int64, (cap, K), "recv_topk_idx", nullable=True),
             _t(disp.get("recv_topk_w"), torch.float32, (cap, K), "recv_topk_w", nullable=True),
             _t(disp.get("recv_src_info"), torch.int32, (cap, 2), "recv_src_info", nullable=True)])


def ep_layout_notify_dispatch(shape: EpShape, x, topk_idx, topk_w, layout: dict, outs: dict, workspace,
                              disp: dict, status, sched=None, host_num_recv_tokens=None, stream=None) -> None:
    """Layout, notify and dispatch in one launch.  ``layout``/``outs`` as for
    :func:`ep_layout_notify`, ``disp`` holds the receive arrays (see
    :func:`alloc_dispatch`; recv_topk_idx / recv_topk_w / recv_src_info may be
    missing or None, and topk_w None with them)."""
    args = _lnd_args(shape, x, topk_idx, topk_w, layout, outs, workspace, disp, sched)
    rc = lib().ep_layout_notify_dispatch(ctypes.byref(shape), *args, _t(status, torch.int32, (1,), "status"),
                                         _sched(sched), _host_counts(shape, host_num_recv_tokens), _stream(stream))
    _check("ep_layout_notify_dispatch", rc)


def ep_debug_layout_notify_dispatch_stall(shape: EpShape, x, topk_idx, topk_w, layout: dict, outs: dict,
                                          workspace, disp: dict, status, stall_tile: int, wait_limit_us: int,
                                          sched=None, stream=None) -> None:
    """Testing hook: :func:`ep_layout_notify_dispatch` with one layout + notify
    tile withholding its lookback words and every wait bounded."""
    args = _lnd_args(shape, x, topk_idx, topk_w, layout, outs, workspace, disp, sched)
    rc = lib().ep_debug_layout_notify_dispatch_stall(
        ctypes.byref(shape), *args, _t(status, torch.int32, (1,), "status"), _sched(sched), _i32(stall_tile),
        _i32(wait_limit_us), _stream(stream))
    _check("ep_debug_layout_notify_dispatch_stall", rc)


def ep_dispatch(shape: EpShape, x, topk_idx, topk_w, send_pos, recv_base, recv_x, recv_topk_idx,
                recv_topk_w, recv_src_info, status, stream=None, sched=None) -> None:
    """Cached mode: pass topk_idx, topk_w, recv_topk_idx and recv_topk_w as None
    (and recv_src_info optionally) to reuse an earlier notify handle.  ``sched``: an
    int64 CUDA tensor of one element, zero before the first call (the calls keep it
    zero), for dynamic assignment of row parts to CTAs; None keeps the static split."""
    R, T, K, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.hidden
    cap = _rows(recv_x, "recv_x")
    rc = lib().ep_dispatch(
        ctypes.byref(shape), _t(x, torch.bfloat16, (R, T, H), "x"),
        _t(topk_idx, torch.int64, (R, T, K), "topk_idx", nullable=True),
        _t(topk_w, torch.float32, (R, T, K), "topk_w", nullable=True),
        _t(send_pos, torch.int32, (R, T, R), "send_pos"),
        _t(recv_base, torch.int64, (R + 1,), "recv_base"), _i64(cap),
        _t(recv_x, torch.bfloat16, (cap, H), "recv_x"),
        _t(recv_topk_idx, torch.int64, (cap, K), "recv_topk_idx", nullable=True),
        _t(recv_topk_w, torch.float32, (cap, K), "recv_topk_w", nullable=True),
        _t(recv_src_info, torch.int32, (cap, 2), "recv_src_info", nullable=True),
        _t(status, torch.int32, (1,), "status"), _sched(sched), _stream(stream))
    _check("ep_dispatch", rc)


def ep_debug_dispatch_stall(shape: EpShape, x, topk_idx, topk_w, send_pos, recv_base, recv_x, recv_topk_idx,
                            recv_topk_w, recv_src_info, status, stall_cta: int, wait_limit_us: int,
                            stream=None, sched=None) -> None:
    """Testing hook: ep_dispatch with CTA ``stall_cta`` never freeing a ring slot and
    every device wait bounded by ``wait_limit_us``; the status word then reports a
    timeout and the context stays usable."""
    R, T, K, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.hidden
    cap = _rows(recv_x, "recv_x")
    rc = lib().ep_debug_dispatch_stall(
        ctypes.byref(shape), _t(x, torch.bfloat16, (R, T, H), "x"),
        _t(topk_idx, torch.int64, (R, T, K), "topk_idx"), _t(topk_w, torch.float32, (R, T, K), "topk_w"),
        _t(send_pos, torch.int32, (R, T, R), "send_pos"), _t(recv_base, torch.int64, (R + 1,), "recv_base"),
        _i64(cap), _t(recv_x, torch.bfloat16, (cap, H), "recv_x"),
        _t(recv_topk_idx, torch.int64, (cap, K), "recv_topk_idx"),
        _t(recv_topk_w, torch.float32, (cap, K), "recv_topk_w"),
        _t(recv_src_info, torch.int32, (cap, 2), "recv_src_info"), _t(status, torch.int32, (1,), "status"),
        _sched(sched), _i32(stall_cta), _i32(wait_limit_us), _stream(stream))
    _check("ep_debug_dispatch_stall", rc)


def ep_dispatch_fp8(shape: EpShape, x, x_scales, topk_idx, topk_w, send_pos, recv_base, recv_x,
                    recv_x_scales, recv_topk_idx, recv_topk_w, recv_src_info, status, stream=None,
                    sched=None) -> None:
    """FP8 rows (uint8 e4m3 bytes, H per token) plus per-token fp32 scales
    ([..., num_scales]; None for none).  Top-k, source info and ``sched`` as in
    ep_dispatch."""
    R, T, K, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.hidden
    cap = _rows(recv_x, "recv_x")
    S = 0 if x_scales is None else x_scales.shape[-1]
    rc = lib().ep_dispatch_fp8(
        ctypes.byref(shape), _t(x, torch.uint8, (R, T, H), "x"),
        _t(x_scales, torch.float32, (R, T, S), "x_scales", nullable=True), _i32(S),
        _t(topk_idx, torch.int64, (R, T, K), "topk_idx", nullable=True),
        _t(topk_w, torch.float32, (R, T, K), "topk_w", nullable=True),
        _t(send_pos, torch.int32, (R, T, R), "send_pos"),
        _t(recv_base, torch.int64, (R + 1,), "recv_base"), _i64(cap),
        _t(recv_x, torch.uint8, (cap, H), "recv_x"),
        _t(recv_x_scales, torch.float32, (cap, S), "recv_x_scales", nullable=True),
        _t(recv_topk_idx, torch.int64, (cap, K), "recv_topk_idx", nullable=True),
        _t(recv_topk_w, torch.float32, (cap, K), "recv_topk_w", nullable=True),
        _t(recv_src_info, torch.int32, (cap, 2), "recv_src_info", nullable=True),
        _t(status, torch.int32, (1,), "status"), _sched(sched), _stream(stream))
    _check("ep_dispatch_fp8", rc)


def ep_combine(shape: EpShape, y, y_w, send_pos, recv_base, combined_x, combined_w, status,
               stream=None) -> None:
    R, T, K, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.hidden
    rows = _rows(y, "y")
    rc = lib().ep_combine(
        ctypes.byref(shape), _t(y, torch.bfloat16, (rows, H), "y"),
        _t(y_w, torch.float32, (rows, K), "y_w", nullable=True), _i64(rows),
        _t(send_pos, torch.int32, (R, T, R), "send_pos"),
        _t(recv_base, torch.int64, (R + 1,), "recv_base"),
        _t(combined_x, torch.bfloat16, (R, T, H), "combined_x"),
        _t(combined_w, torch.float32, (R, T, K), "combined_w", nullable=True),
        _t(status, torch.int32, (1,), "status"), _stream(stream))
    _check("ep_combine", rc)


def ep_ll_layout(shape: EpShape, topk_idx, num_tokens_per_expert, expert_capacity: int, slot_pos,
                 layout_range, count, status, stream=None) -> None:
    """Low-latency (per-expert packed) layout: row of each slot in its expert's buffer.
    ``num_tokens_per_expert`` may be None: the kernel then counts for itself (R <= 16)."""
    R, T, K, E = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.num_experts
    rc = lib().ep_ll_layout(
        ctypes.byref(shape), _t(topk_idx, torch.int64, (R, T, K), "topk_idx"),
        _t(num_tokens_per_expert, torch.int32, (R, E), "num_tokens_per_expert", nullable=True),
        _i32(expert_capacity),
        _t(slot_pos, torch.int32, (R, T, K), "slot_pos"), _t(layout_range, torch.int32, (E, R, 2), "layout_range"),
        _t(count, torch.int32, (E,), "count"), _t(status, torch.int32, (1,), "status"), _stream(stream))
    _check("ep_ll_layout", rc)


def ep_ll_dispatch(shape: EpShape, x, topk_idx, slot_pos, expert_capacity: int, recv_x, recv_src_info,
                   status, stream=None, sched=None) -> None:
    R, T, K, E, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.num_experts, shape.hidden
    cap = expert_capacity
    rc = lib().ep_ll_dispatch(
        ctypes.byref(shape), _t(x, torch.bfloat16, (R, T, H), "x"),
        _t(topk_idx, torch.int64, (R, T, K), "topk_idx"), _t(slot_pos, torch.int32, (R, T, K), "slot_pos"),
        _i32(cap), _t(recv_x, torch.bfloat16, (E, cap, H), "recv_x"),
        _t(recv_src_info, torch.int32, (E, cap, 2), "recv_src_info", nullable=True),
        _t(status, torch.int32, (1,), "status"), _sched(sched), _stream(stream))
    _check("ep_ll_dispatch", rc)


def ep_ll_combine(shape: EpShape, y, expert_capacity: int, topk_idx, topk_w, slot_pos, combined_x, status,
                  stream=None) -> None:
    R, T, K, E, H = shape.num_ranks, shape.num_tokens, shape.num_topk, shape.num_experts, shape.hidden
    cap = expert_capacity
    rc = lib().ep_ll_combine(
        ctypes.byref(shape), _t(y, torch.bfloat16, (E, cap, H), "y"), _i32(cap),
        _t(topk_idx, torch.int64, (R, T, K), "topk_idx"), _t(topk_w, torch.float32, (R, T, K), "topk_w"),
        _t(slot_pos, torch.int32, (R, T, K), "slot_pos"), _t(combined_x, torch.bfloat16, (R, T, H), "combined_x"),
        _t(status, torch.int32, (1,), "status"), _stream(stream))
    _check("ep_ll_combine", rc)


def ep_sync_status(status, stream=None) -> int:
    """Wait for the stream and return the status code the device word maps to."""
    return int(lib().ep_sync_status(_t(status, torch.int32, (1,), "status"), _stream(stream)))


# --------------------------------------------------------------------------- allocation
def alloc_layout(shape: EpShape, device="cuda") -> dict:
    R, T, E, N = shape.num_ranks, shape.num_tokens, shape.num_experts, shape.N
    z = lambda *s, dt=torch.int32: torch.empty(s, dtype=dt, device=device)  # noqa: E731
    return dict(num_tokens_per_rank=z(R, R), num_tokens_per_rdma_rank=z(R, N),
                num_tokens_per_expert=z(R, E), is_token_in_rank=z(R, T, R, dt=torch.uint8))


def alloc_notify(shape: EpShape, device="cuda") -> dict:
    outs = {k: torch.empty(s, dtype=dt, device=device) for k, (s, dt) in notify_shapes(shape).items()}
    ws = ep_notify_workspace_bytes(shape)
    # zeroed once here; every notify call leaves it ready for the next one
    outs["workspace"] = torch.zeros((ws + 15) // 16 * 16, dtype=torch.uint8, device=device)
    return outs


def alloc_layout_notify_workspace(shape: EpShape, device="cuda", nbytes: int | None = None) -> torch.Tensor:
    """Zeroed workspace for :func:`ep_layout_notify` (every call leaves it ready
    for the next one); ``nbytes`` overrides the size (e.g. for several shapes)."""
    n = ep_layout_notify_workspace_bytes(shape) if nbytes is None else nbytes
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def alloc_dispatch(shape: EpShape, capacity_rows: int, device="cuda") -> dict:
    H, K = shape.hidden, shape.num_topk
    return dict(recv_x=torch.empty(capacity_rows, H, dtype=torch.bfloat16, device=device),
                recv_topk_idx=torch.empty(capacity_rows, K, dtype=torch.int64, device=device),
                recv_topk_w=torch.empty(capacity_rows, K, dtype=torch.float32, device=device),
                recv_src_info=torch.empty(capacity_rows, 2, dtype=torch.int32, device=device))


def alloc_combine(shape: EpShape, device="cuda") -> dict:
    R, T, H, K = shape.num_ranks, shape.num_tokens, shape.hidden, shape.num_topk
    return dict(combined_x=torch.empty(R, T, H, dtype=torch.bfloat16, device=device),
                combined_w=torch.empty(R, T, K, dtype=torch.float32, device=device))


@dataclass
class Pipeline:
    """Buffers for one shape plus the four steps in order (identity expert by
    default).  Allocates once; :meth:`run` launches layout + notify (one call,
    :func:`ep_layout_notify`), dispatch and combine on the current stream
    without synchronising."""

    shape: EpShape
    capacity_rows: int
    device: str = "cuda"

    def __post_init__(self):
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        # dispatch's unit counter: zeroed once here, every call leaves it zero
        self.sched = torch.zeros(1, dtype=torch.int64, device=self.device)
        self.layout = alloc_layout(self.shape, self.device)
        self.notify = alloc_notify(self.shape, self.device)
        self.ln_workspace = alloc_layout_notify_workspace(self.shape, self.device)
        self.dispatch = alloc_dispatch(self.shape, self.capacity_rows, self.device)
        self.combine = alloc_combine(self.shape, self.device)

    def run(self, x, topk_idx, topk_w, y=None, y_w=None, stream=None, host_num_recv_tokens=None):
        sh, L, Nt, D, C = self.shape, self.layout, self.notify, self.dispatch, self.combine
        ep_layout_notify(sh, topk_idx, L, Nt, self.ln_workspace, self.status, host_num_recv_tokens, stream)
        ep_dispatch(sh, x, topk_idx, topk_w, Nt["send_pos"], Nt["recv_base"], D["recv_x"],
                    D["recv_topk_idx"], D["recv_topk_w"], D["recv_src_info"], self.status, stream, self.sched)
        ep_combine(sh, D["recv_x"] if y is None else y, D["recv_topk_w"] if y_w is None else y_w,
                   Nt["send_pos"], Nt["recv_base"], C["combined_x"], C["combined_w"], self.status,
                   stream)
        return C["combined_x"], C["combined_w"]

    def run_cached(self, x, y=None, stream=None):
        """Cached mode: dispatch and combine only, reusing the handle (send_pos,
        recv_base) of the last :meth:`run`; the top-k is not dispatched and the
        combined weights are not produced."""
        sh, Nt, D, C = self.shape, self.notify, self.dispatch, self.combine
        ep_dispatch(sh, x, None, None, Nt["send_pos"], Nt["recv_base"], D["recv_x"], None, None, None,
                    self.status, stream, self.sched)
        ep_combine(sh, D["recv_x"] if y is None else y, None, Nt["send_pos"], Nt["recv_base"],
                   C["combined_x"], None, self.status, stream)
        return C["combined_x"]
