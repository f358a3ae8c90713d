"""CPU oracle for the MoE dispatch/combine hot path (test infrastructure).

This package is test infrastructure, not part of the product.  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import it.  The arithmetic lives in ``ep_oracle.c`` (plain C, single thread);
this module compiles it with gcc on first use and wraps it with ctypes and
numpy.  Each wrapper names the step it follows; the C file cites the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()

NODE_SIZE = 8


def build(mutant: int = 0) -> str:
    """Compile the oracle into ``oracle/_build``; return the .so path.

    ``mutant`` > 0 compiles a copy with a planted mistake (see
    ``ORACLE_MUTANT`` in the C file) for the tests that show the pins catch it.
    """
    os.makedirs(_BUILD, exist_ok=True)
    name = "libep_oracle.so" if mutant == 0 else f"libep_oracle_mutant{mutant}.so"
    out = os.path.join(_BUILD, name)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp]
    subprocess.check_call(cmd + ["-lm"])
    os.replace(tmp, out)
    return out


def _p(a: np.ndarray):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.lib = ctypes.CDLL(path)
        for fn in ("oracle_layout", "oracle_notify", "oracle_dispatch", "oracle_dispatch_fp8",
                   "oracle_combine", "oracle_num_nodes", "oracle_ll_layout", "oracle_ll_dispatch",
                   "oracle_ll_combine"):
            getattr(self.lib, fn).restype = ctypes.c_int
        self.lib.oracle_f32_to_bf16.restype = None

    # -- helpers -----------------------------------------------------------------
    def num_nodes(self, R: int) -> int:
        return int(self.lib.oracle_num_nodes(ctypes.c_int(R)))

    def f32_to_bf16(self, a: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(a, dtype=np.float32)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_bf16(_p(a), _p(out), ctypes.c_int64(a.size))
        return out

    # -- step 1 --------------------------------------------------------------------
    def layout(self, R, T, K, E, topk_idx):
        """Layout counting (getDispatchLayout)."""
        N = self.num_nodes(R)
        topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64).reshape(R, T, K)
        out = dict(
            num_tokens_per_rank=np.zeros((R, R), np.int32),
            num_tokens_per_rdma_rank=np.zeros((R, N), np.int32),
            num_tokens_per_expert=np.zeros((R, E), np.int32),
            is_token_in_rank=np.zeros((R, T, R), np.uint8),
        )
        rc = self.lib.oracle_layout(R, T, K, E, _p(topk_idx), _p(out["num_tokens_per_rank"]),
                                    _p(out["num_tokens_per_rdma_rank"]),
                                    _p(out["num_tokens_per_expert"]), _p(out["is_token_in_rank"]))
        if rc != 0:
            raise ValueError("oracle_layout: expert id outside [-1, E)")
        return out

    # -- step 2 --------------------------------------------------------------------
    def notify(self, R, T, E, C, expert_alignment, layout):
        """Notify prefix sums (notify_dispatch) from the layout outputs."""
        N = self.num_nodes(R)
        E_loc = E // R
        ins = [np.ascontiguousarray(layout[k]) for k in
               ("is_token_in_rank", "num_tokens_per_rank", "num_tokens_per_rdma_rank",
                "num_tokens_per_expert")]
        out = dict(
            rank_prefix_matrix=np.zeros((R, R), np.int32),
            gbl_channel_prefix_matrix=np.zeros((R, R, C), np.int32),
            rdma_channel_prefix_matrix=np.zeros((R, N, C), np.int32),
            recv_gbl_rank_prefix_sum=np.zeros((R, R), np.int32),
            recv_rdma_rank_prefix_sum=np.zeros((R, N), np.int32),
            recv_channel_offset=np.zeros((R, R, C), np.int32),
            num_recv_tokens=np.zeros((R,), np.int32),
            num_rdma_recv_tokens=np.zeros((R,), np.int32),
            num_recv_tokens_per_expert=np.zeros((R, E_loc), np.int32),
            recv_base=np.zeros((R + 1,), np.int64),
            send_pos=np.zeros((R, T, R), np.int32),
        )
        order = ("rank_prefix_matrix", "gbl_channel_prefix_matrix", "rdma_channel_prefix_matrix",
                 "recv_gbl_rank_prefix_sum", "recv_rdma_rank_prefix_sum", "recv_channel_offset",
                 "num_recv_tokens", "num_rdma_recv_tokens", "num_recv_tokens_per_expert",
                 "recv_base", "send_pos")
        rc = self.lib.oracle_notify(R, T, E, C, expert_alignment, *[_p(a) for a in ins],
                                    *[_p(out[k]) for k in order])
        if rc != 0:
            raise ValueError("oracle_notify: bad arguments")
        return out

    # -- step 3 --------------------------------------------------------------------
    def dispatch(self, R, T, K, E, H, C, x, topk_idx, topk_w, send_pos, recv_base, payload=True,
                 with_topk=True):
        """Dispatch; ``payload=False`` computes only the metadata rows;
        ``with_topk=False`` is cached mode (no top-k fields)."""
        rows = int(recv_base[-1])
        topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
        topk_w = np.ascontiguousarray(topk_w, dtype=np.float32)
        send_pos = np.ascontiguousarray(send_pos, dtype=np.int32)
        recv_base = np.ascontiguousarray(recv_base, dtype=np.int64)
        out = dict(
            recv_x=np.zeros((rows, H), np.uint16) if payload else None,
            recv_topk_idx=np.zeros((rows, K), np.int64) if with_topk else None,
            recv_topk_w=np.zeros((rows, K), np.float32) if with_topk else None,
            recv_src_info=np.zeros((rows, 2), np.int32),
        )
        xs = np.ascontiguousarray(x, dtype=np.uint16) if payload else None
        rc = self.lib.oracle_dispatch(R, T, K, E, H, C, _p(xs), _p(topk_idx), _p(topk_w),
                                      _p(send_pos), _p(recv_base), _p(out["recv_x"]),
                                      _p(out["recv_topk_idx"]), _p(out["recv_topk_w"]),
                                      _p(out["recv_src_info"]))
        if rc != 0:
            raise ValueError("oracle_dispatch: a row falls outside its destination region")
        return out

    def dispatch_fp8(self, R, T, K, E, H, C, x, x_scales, topk_idx, topk_w, send_pos, recv_base,
                     with_topk=True):
        """FP8 dispatch: byte rows (H per token) plus their fp32 scales rows."""
        rows = int(recv_base[-1])
        S = 0 if x_scales is None else int(x_scales.shape[-1])
        x = np.ascontiguousarray(x, dtype=np.uint8)
        xs = None if x_scales is None else np.ascontiguousarray(x_scales, dtype=np.float32)
        ti = np.ascontiguousarray(topk_idx, dtype=np.int64) if with_topk else None
        tw = np.ascontiguousarray(topk_w, dtype=np.float32) if with_topk else None
        out = dict(
            recv_x=np.zeros((rows, H), np.uint8),
            recv_x_scales=np.zeros((rows, S), np.float32) if S else None,
            recv_topk_idx=np.zeros((rows, K), np.int64) if with_topk else None,
            recv_topk_w=np.zeros((rows, K), np.float32) if with_topk else None,
            recv_src_info=np.zeros((rows, 2), np.int32),
        )
        rc = self.lib.oracle_dispatch_fp8(R, T, K, E, H, C, S, _p(x), _p(xs), _p(ti), _p(tw),
                                          _p(np.ascontiguousarray(send_pos, dtype=np.int32)),
                                          _p(np.ascontiguousarray(recv_base, dtype=np.int64)),
                                          _p(out["recv_x"]), _p(out["recv_x_scales"]),
                                          _p(out["recv_topk_idx"]), _p(out["recv_topk_w"]),
                                          _p(out["recv_src_info"]))
        if rc != 0:
            raise ValueError("oracle_dispatch_fp8: a row falls outside its destination region")
        return out

    # -- step 4 --------------------------------------------------------------------
    def combine(self, R, T, K, H, y, y_w, send_pos, recv_base):
        """Combine: fp32 sum in ascending rank order, bf16 round to nearest even."""
        y = np.ascontiguousarray(y, dtype=np.uint16).reshape(-1, H)
        y_w = None if y_w is None else np.ascontiguousarray(y_w, dtype=np.float32).reshape(-1, K)
        assert y_w is None or y_w.shape[0] == y.shape[0], "y and y_w must have the same rows"
        send_pos = np.ascontiguousarray(send_pos, dtype=np.int32)
        recv_base = np.ascontiguousarray(recv_base, dtype=np.int64)
        cx = np.zeros((R, T, H), np.uint16)
        cw = np.zeros((R, T, K), np.float32) if y_w is not None else None
        rc = self.lib.oracle_combine(R, T, K, H, ctypes.c_int64(y.shape[0]), _p(y), _p(y_w),
                                     _p(send_pos), _p(recv_base), _p(cx), _p(cw))
        if rc != 0:
            raise ValueError("oracle_combine: a row lies outside y")
        return dict(combined_x=cx, combined_w=cw)


# -- low-latency (per-expert packed) layout -------------------------------------------
def ll_layout(o: "Oracle", R, T, K, E, cap, topk_idx):
    """Row of every slot inside its expert's buffer, per-source ranges, counts."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64).reshape(R, T, K)
    out = dict(slot_pos=np.zeros((R, T, K), np.int32), layout_range=np.zeros((E, R, 2), np.int32),
               count=np.zeros((E,), np.int32))
    rc = o.lib.oracle_ll_layout(R, T, K, E, cap, _p(idx), _p(out["slot_pos"]), _p(out["layout_range"]),
                                _p(out["count"]))
    if rc < 0:
        raise ValueError("oracle_ll_layout: expert id outside [-1, E)")
    out["dropped"] = rc == 1
    return out


def ll_dispatch(o: "Oracle", R, T, K, E, H, cap, x, topk_idx, slot_pos):
    recv_x = np.zeros((E, cap, H), np.uint16)
    src = np.full((E, cap, 2), -1, np.int32)
    rc = o.lib.oracle_ll_dispatch(R, T, K, E, H, cap, _p(np.ascontiguousarray(x, dtype=np.uint16)),
                                  _p(np.ascontiguousarray(topk_idx, dtype=np.int64)),
                                  _p(np.ascontiguousarray(slot_pos, dtype=np.int32)), _p(recv_x), _p(src))
    if rc != 0:
        raise ValueError("oracle_ll_dispatch: row outside its buffer")
    return dict(recv_x=recv_x, recv_src_info=src)


def ll_combine(o: "Oracle", R, T, K, E, H, cap, y, topk_idx, topk_w, slot_pos):
    out = np.zeros((R, T, H), np.uint16)
    rc = o.lib.oracle_ll_combine(R, T, K, E, H, cap, _p(np.ascontiguousarray(y, dtype=np.uint16)),
                                 _p(np.ascontiguousarray(topk_idx, dtype=np.int64)),
                                 _p(np.ascontiguousarray(topk_w, dtype=np.float32)),
                                 _p(np.ascontiguousarray(slot_pos, dtype=np.int32)), _p(out))
    if rc != 0:
        raise ValueError("oracle_ll_combine: row outside its buffer")
    return out


def load(mutant: int = 0) -> Oracle:
    """Build (if needed) and load the oracle library."""
    global _LIB
    with _LOCK:
        if mutant:
            return Oracle(build(mutant))
        if _LIB is None:
            _LIB = Oracle(build())
        return _LIB


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 values (exact)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_all(R, T, K, E, H, C, expert_alignment, x, topk_idx, topk_w, oracle: Oracle | None = None):
    """The whole path with the identity expert: layout, notify, dispatch, combine."""
    o = oracle or load()
    lay = o.layout(R, T, K, E, topk_idx)
    nt = o.notify(R, T, E, C, expert_alignment, lay)
    dp = o.dispatch(R, T, K, E, H, C, x, topk_idx, topk_w, nt["send_pos"], nt["recv_base"])
    cb = o.combine(R, T, K, H, dp["recv_x"], dp["recv_topk_w"], nt["send_pos"], nt["recv_base"])
    return lay, nt, dp, cb
