"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import Workload, gen_routing, gen_x


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its bit patterns as uint16 (host)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_equal(name: str, got: np.ndarray, want: np.ndarray) -> None:
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{name}: shape {got.shape} != {want.shape}"
    if got.dtype.kind == "f":
        eq = (got.view(np.uint32 if got.itemsize == 4 else np.uint64) ==
              want.view(np.uint32 if want.itemsize == 4 else np.uint64))
    else:
        eq = got == want
    if not eq.all():
        bad = np.argwhere(~eq)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches; first at {i}: got {got[i]!r}, "
                             f"want {want[i]!r}")


def assert_combine_close(name: str, got_bits: np.ndarray, want_bits: np.ndarray) -> None:
    """The combine contract: |got - ref| <= 1e-2 + 8e-3 |ref|; also report exactness."""
    g = oracle.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = oracle.bf16_bits_to_f32(want_bits).astype(np.float64)
    err = np.abs(g - r)
    tol = 1e-2 + 8e-3 * np.abs(r)
    if not (err <= tol).all():
        bad = np.argwhere(~(err <= tol))
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} outside tolerance; first at {i}: got {g[i]}, "
                             f"want {r[i]}")
    # The kernel sums in the same order with the same fp32 operations, so the
    # bits are expected to agree exactly as well.
    assert_equal(name + " (bits)", got_bits, want_bits)


def shape_of(w: Workload) -> ep.EpShape:
    return ep.EpShape.make(w.R, w.T, w.K, w.E, w.H, w.C, w.expert_alignment)


def make_inputs(w: Workload, x_on_gpu: bool = False):
    idx, wt = gen_routing(w)
    x = gen_x(w, "cuda" if x_on_gpu else "cpu")
    return idx, wt, x


def run_layout_notify(w: Workload, idx: torch.Tensor, status=None):
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    ep.ep_notify_dispatch(sh, lay["is_token_in_rank"], lay["num_tokens_per_rank"],
                          lay["num_tokens_per_rdma_rank"], lay["num_tokens_per_expert"], nt,
                          nt["workspace"], status)
    return sh, lay, nt, status


LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_rdma_rank", "num_tokens_per_expert",
               "is_token_in_rank")
NOTIFY_KEYS = ("rank_prefix_matrix", "gbl_channel_prefix_matrix", "rdma_channel_prefix_matrix",
               "recv_gbl_rank_prefix_sum", "recv_rdma_rank_prefix_sum", "recv_channel_offset",
               "num_recv_tokens", "num_rdma_recv_tokens", "num_recv_tokens_per_expert", "recv_base",
               "send_pos")


def check_layout_notify(lay_gpu, nt_gpu, lay_ref, nt_ref):
    for k in LAYOUT_KEYS:
        assert_equal(k, lay_gpu[k].cpu().numpy(), lay_ref[k])
    for k in NOTIFY_KEYS:
        assert_equal(k, nt_gpu[k].cpu().numpy(), nt_ref[k])
