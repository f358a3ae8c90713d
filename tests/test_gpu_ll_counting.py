"""ep_ll_layout without the per-expert count input (one thread-block cluster
counts and exchanges the per-source totals itself) vs the CPU oracle, bit-exact,
through the C ABI; and the shapes it refuses."""
from __future__ import annotations

import pytest
import torch

import oracle
from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import CONFIGS, Workload, gen_routing
from gpu_util import assert_equal, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.lib()


CASES = {
    "tiny": (CONFIGS["tiny"], 1),
    "low_latency": (CONFIGS["low_latency"], 1),
    "single_rank": (Workload("e", R=1, T=37, H=64, E=6, K=3, C=4, routing="replace", mask=0.2), 1),
    "repeats_r16": (Workload("e", R=16, T=50, H=64, E=64, K=8, C=3, routing="replace", mask=0.3), None),
    "odd_ranks_odd_k": (Workload("e", R=3, T=41, H=72, E=9, K=5, C=5, mask=0.1), 1),
    "zipf_r8": (Workload("e", R=8, T=1000, H=64, E=256, K=8, C=4, routing="zipf"), 1),
    "max_exchange": (Workload("e", R=16, T=64, H=64, E=1024, K=4, C=2), 1),  # R*E = 16384
    "empty_tokens": (Workload("e", R=4, T=0, H=64, E=8, K=2, C=3), 1),
    "capacity_drop": (CONFIGS["tiny"], 0),
}


def _run(w, cap, idx, counts):
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slot = torch.full((w.R, w.T, w.K), -7, dtype=torch.int32, device="cuda")
    rng_ = torch.full((w.E, w.R, 2), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((w.E,), -7, dtype=torch.int32, device="cuda")
    ep.ep_ll_layout(sh, idx.cuda(), counts, cap, slot, rng_, cnt, status)
    return status, slot, rng_, cnt


@pytest.mark.parametrize("name", sorted(CASES))
def test_ll_layout_counting_form_matches_oracle(name):
    w, capf = CASES[name]
    cap = 7 if capf == 0 else w.R * w.T * (capf or w.K)
    idx, _ = gen_routing(w)
    o = oracle.load()
    ref = oracle.ll_layout(o, w.R, w.T, w.K, w.E, cap, idx.numpy())
    status, slot, rng_, cnt = _run(w, cap, idx, None)
    want = ep.EP_ERR_CAPACITY if ref["dropped"] else ep.EP_OK
    assert ep.ep_sync_status(status) == want
    assert_equal("ll slot_pos", slot.cpu().numpy(), ref["slot_pos"])
    assert_equal("ll layout_range", rng_.cpu().numpy(), ref["layout_range"])
    assert_equal("ll count", cnt.cpu().numpy(), ref["count"])
    # and the same as the form that takes the counts from the layout step
    sh = shape_of(w)
    lay = ep.alloc_layout(sh)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], st2)
    st3, slot2, rng2, cnt2 = _run(w, cap, idx, lay["num_tokens_per_expert"])
    assert ep.ep_sync_status(st3) == want
    assert torch.equal(slot, slot2) and torch.equal(rng_, rng2) and torch.equal(cnt, cnt2)


@pytest.mark.parametrize("R,E", [(32, 256), (16, 2048)])
def test_ll_layout_counting_form_refuses_large_shapes(R, E):
    w = Workload("e", R=R, T=8, H=64, E=E, K=2, C=1)
    sh = shape_of(w)
    idx, _ = gen_routing(w)
    with pytest.raises(ep.EpError) as exc:
        _run(w, 16, idx, None)
    assert exc.value.status == ep.EP_ERR_INVALID_ARG
    assert sh.num_ranks == R


def test_ll_layout_counting_form_reports_bad_ids():
    w = Workload("e", R=8, T=33, H=64, E=64, K=4, C=2)
    idx, _ = gen_routing(w)
    idx[2, 7, 1] = w.E
    idx[5, 0, 3] = -9
    status, slot, rng_, cnt = _run(w, w.R * w.T, idx, None)
    assert ep.ep_sync_status(status) == ep.EP_ERR_INPUT
    clean = idx.clone()
    clean[2, 7, 1] = -1
    clean[5, 0, 3] = -1
    ref = oracle.ll_layout(oracle.load(), w.R, w.T, w.K, w.E, w.R * w.T, clean.numpy())
    assert_equal("ll slot_pos (bad ids ignored)", slot.cpu().numpy(), ref["slot_pos"])
    assert_equal("ll count (bad ids ignored)", cnt.cpu().numpy(), ref["count"])
