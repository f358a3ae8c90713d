"""The one-launch forms of layout + notify agree with the separate calls on
random shapes: 200 seeded shapes (ranks, tokens, experts, top-k, channels,
routing, masking, alignment), each run through ep_get_dispatch_layout +
ep_notify_dispatch (checked against the CPU oracle by the parity suites), the
tiled form with a random tile size, ep_layout_notify's default form and the
one-launch layout + notify + dispatch, all of the tiled and fused calls on
ONE shared workspace (so calls of changing shapes and tile counts follow each
other on it); every layout and notify output, and every dispatched row and
field of the one-launch dispatch (against ep_dispatch on the separate calls'
row map), bit-exact."""
from __future__ import annotations

import random

import pytest
import torch

from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import Workload, gen_routing, gen_x, worst_case_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.lib()


def _random_workload(rng: random.Random, i: int) -> Workload:
    R = rng.choice([1, 2, 3, 4, 6, 8, 16, 24, 32])
    E = R * rng.choice([1, 2, 4, 8, 16])
    K = min(rng.choice([1, 2, 3, 4, 6, 8]), E)
    T = rng.choice([0, 1, 5, 31, 32, 33, 100, 511, 512, 513, 1000, 2048, 3000, 4096])
    T = min(T, 65536 // R)
    return Workload("agree", R=R, T=T, H=64, E=E, K=K, C=rng.choice([1, 3, 8, 24]),
                    routing=rng.choice(["uniform", "zipf", "replace"]), mask=rng.choice([0.0, 0.1, 0.5]),
                    seed=i, expert_alignment=rng.choice([1, 1, 4]))


def test_forms_agree_on_random_shapes():
    dev = torch.device("cuda")
    rng = random.Random(2024)
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=dev)
    for i in range(200):
        w = _random_workload(rng, i)
        sh = ep.EpShape.make(w.R, w.T, w.K, w.E, w.H, w.C, w.expert_alignment)
        idx, wt = gen_routing(w)
        idx, wt = idx.to(dev), wt.to(dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        lay0, nt0 = ep.alloc_layout(sh), ep.alloc_notify(sh)
        ep.ep_get_dispatch_layout(sh, idx, lay0["num_tokens_per_rank"], lay0["num_tokens_per_rdma_rank"],
                                  lay0["num_tokens_per_expert"], lay0["is_token_in_rank"], st)
        ep.ep_notify_dispatch(sh, lay0["is_token_in_rank"], lay0["num_tokens_per_rank"],
                              lay0["num_tokens_per_rdma_rank"], lay0["num_tokens_per_expert"], nt0, nt0["workspace"], st)
        forms = []
        tile = rng.choice([0, 0, 32, 64, 96, 128, 256, 512])
        lay1, nt1 = ep.alloc_layout(sh), ep.alloc_notify(sh)
        ep.ep_debug_layout_notify_tiled(sh, idx, lay1, nt1, ws, st, tile_tokens=tile)
        forms.append((f"tiled, {tile}-token tiles", lay1, nt1))
        lay2, nt2 = ep.alloc_layout(sh), ep.alloc_notify(sh)
        ep.ep_layout_notify(sh, idx, lay2, nt2, ws, st)
        forms.append(("ep_layout_notify", lay2, nt2))
        disp = None
        if w.T > 0:
            x = gen_x(w, dev)
            lay3, nt3 = ep.alloc_layout(sh), ep.alloc_notify(sh)
            disp = ep.alloc_dispatch(sh, max(1, worst_case_rows(w)))
            ep.ep_layout_notify_dispatch(sh, x, idx, wt, lay3, nt3, ws, disp, st)
            forms.append(("ep_layout_notify_dispatch", lay3, nt3))
            ref = ep.alloc_dispatch(sh, max(1, worst_case_rows(w)))
            ep.ep_dispatch(sh, x, idx, wt, nt0["send_pos"], nt0["recv_base"], ref["recv_x"], ref["recv_topk_idx"],
                           ref["recv_topk_w"], ref["recv_src_info"], st)
        assert ep.ep_sync_status(st) == ep.EP_OK, w
        for name, lay, nt in forms:
            for k in lay0:
                assert torch.equal(lay[k], lay0[k]), (name, k, w)
            for k in nt0:
                if k != "workspace":
                    assert torch.equal(nt[k], nt0[k]), (name, k, w)
        if disp is not None:
            rows = int(nt0["recv_base"][-1].item())
            for k in ("recv_x", "recv_topk_idx", "recv_topk_w", "recv_src_info"):
                a, b = disp[k][:rows], ref[k][:rows]
                if a.dtype == torch.bfloat16:
                    a, b = a.view(torch.int16), b.view(torch.int16)
                assert torch.equal(a, b), ("one-launch dispatch", k, w)
