"""ep_layout_notify_dispatch (layout, notify and dispatch in one launch) vs the
CPU oracle, element by element, through the C ABI: every layout and notify
output and every dispatched row, top-k field and source-info pair, bit-exact,
with the static split and with the run-time unit counter; at full size
(skewed, large) compared with the separate calls; plus the cases without
top-k fields, the stalled tile, first call inside a CUDA-graph capture and a
workspace shared with ep_layout_notify."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import CONFIGS, Workload, gen_routing, gen_x, worst_case_rows
from gpu_util import assert_equal, check_layout_notify, shape_of, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.lib()


def _buffers(w: Workload, cap: int | None = None, topk: bool = True):
    sh = shape_of(w)
    lay, nt = ep.alloc_layout(sh), ep.alloc_notify(sh)
    for d in (lay, nt):
        for k, v in d.items():
            if k != "workspace":
                v.fill_(0x5A if v.dtype == torch.uint8 else -7)
    disp = ep.alloc_dispatch(sh, max(1, worst_case_rows(w)) if cap is None else cap)
    if not topk:
        disp["recv_topk_idx"] = None
        disp["recv_topk_w"] = None
    return sh, lay, nt, disp


def _oracle_all(w: Workload, idx, wt, x):
    o = oracle.load()
    xb = x.view(torch.int16).numpy().view(np.uint16)
    lay = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay)
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, xb, idx.numpy(), wt.numpy(), nt["send_pos"], nt["recv_base"])
    return lay, nt, dp


def _check_dispatch(disp, dp, rows, topk=True):
    assert_equal("recv_x", u16(disp["recv_x"][:rows]), dp["recv_x"])
    assert_equal("recv_src_info", disp["recv_src_info"][:rows].cpu().numpy(), dp["recv_src_info"])
    if topk:
        assert_equal("recv_topk_idx", disp["recv_topk_idx"][:rows].cpu().numpy(), dp["recv_topk_idx"])
        assert_equal("recv_topk_w", disp["recv_topk_w"][:rows].cpu().numpy(), dp["recv_topk_w"])


CASES = {
    "tiny": CONFIGS["tiny"],
    "low_latency": CONFIGS["low_latency"],
    "prefill": CONFIGS["prefill"],
    "single_rank": Workload("e", R=1, T=37, H=64, E=6, K=3, C=4, routing="replace", mask=0.2),
    "channels_exceed_tokens": Workload("e", R=8, T=50, H=128, E=64, K=4, C=64, mask=0.1),
    "top1": Workload("e", R=16, T=33, H=256, E=64, K=1, C=5),
    "r32_min_hidden_repeats": Workload("e", R=32, T=19, H=8, E=256, K=8, C=3, routing="replace", mask=0.3),
    "all_masked": Workload("e", R=8, T=40, H=64, E=16, K=4, C=4, mask=1.0),
    "ragged_r16_zipf": Workload("e", R=16, T=1001, H=264, E=256, K=7, C=13, routing="zipf", mask=0.05),
    "odd_ranks_align": Workload("e", R=3, T=41, H=72, E=9, K=2, C=5, expert_alignment=4),
    "k32_repeats": Workload("e", R=16, T=97, H=64, E=512, K=32, C=7, routing="replace", mask=0.1),
    "one_token": Workload("e", R=16, T=1, H=64, E=16, K=3, C=1),
    "r24_many_tiles": Workload("e", R=24, T=1500, H=136, E=96, K=6, C=9, mask=0.1),
    # 512 tiles of 512 tokens, more than the grid's CTAs: later tiles by ticket
    "r32_more_tiles_than_ctas": Workload("e", R=32, T=8192, H=64, E=256, K=8, C=16, mask=0.05),
}


@pytest.mark.parametrize("sched", [False, True], ids=["static", "counter"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_matches_oracle(name, sched):
    w = CASES[name]
    idx, wt = gen_routing(w)
    x = gen_x(w)
    lay_ref, nt_ref, dp = _oracle_all(w, idx, wt, x)
    sh, lay, nt, disp = _buffers(w)
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, dtype=torch.int64, device="cuda") if sched else None
    host = torch.full((w.R + 1,), -1, dtype=torch.int32).pin_memory()
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status, sc, host)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    _check_dispatch(disp, dp, int(nt_ref["recv_base"][-1]))
    assert np.array_equal(host.numpy(), np.concatenate([nt_ref["num_recv_tokens"], nt_ref["recv_base"][-1:]]))
    if sc is not None:
        assert int(sc.item()) == 0  # the counter is left zero for the next call
    # a second call on the same buffers and workspace gives byte-identical results
    outs = {**lay, **{k: v for k, v in nt.items() if k != "workspace"},
            "recv_x": disp["recv_x"].view(torch.int16), "recv_src_info": disp["recv_src_info"]}
    snap = {k: v.clone() for k, v in outs.items()}
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status, sc)
    assert ep.ep_sync_status(status) == ep.EP_OK
    for k, v in snap.items():
        assert torch.equal(v, outs[k]), f"{k} differs between calls"


def test_fused_without_topk_fields():
    """topk_w and both top-k receive arrays NULL: rows and source info only."""
    w = CASES["ragged_r16_zipf"]
    idx, wt = gen_routing(w)
    x = gen_x(w)
    lay_ref, nt_ref, dp = _oracle_all(w, idx, wt, x)
    sh, lay, nt, disp = _buffers(w, topk=False)
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), None, lay, nt, ws, disp, status)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    _check_dispatch(disp, dp, int(nt_ref["recv_base"][-1]), topk=False)


def test_fused_empty_tokens_writes_layout_and_notify():
    w = Workload("e", R=4, T=0, H=64, E=8, K=2, C=3)
    idx, wt = gen_routing(w)
    x = gen_x(w)
    lay_ref, nt_ref, _ = _oracle_all(w, idx, wt, x)
    sh, lay, nt, disp = _buffers(w, cap=1)
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)


@pytest.mark.parametrize("name", ["skewed", "large"])
def test_fused_full_size_matches_separate_calls(name):
    """Full size: layout and notify outputs against the oracle, every received
    row and field against the separate calls (ep_layout_notify, ep_dispatch)
    on the same inputs, with the counter as the bench runs it."""
    w = CONFIGS[name]
    o = oracle.load()
    idx, wt = gen_routing(w)
    x = gen_x(w, "cuda")
    lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
    rows = int(nt_ref["recv_base"][-1])
    sh = shape_of(w)
    idx_d, wt_d = idx.cuda(), wt.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = ep.alloc_layout_notify_workspace(sh)
    # separate calls first
    lay1, nt1 = ep.alloc_layout(sh), ep.alloc_notify(sh)
    d1 = ep.alloc_dispatch(sh, rows)
    ep.ep_layout_notify(sh, idx_d, lay1, nt1, ws, status)
    ep.ep_dispatch(sh, x, idx_d, wt_d, nt1["send_pos"], nt1["recv_base"], d1["recv_x"], d1["recv_topk_idx"],
                   d1["recv_topk_w"], d1["recv_src_info"], status, sched=sc)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay1, nt1, lay_ref, nt_ref)
    # the fused call, same workspace
    lay2, nt2 = ep.alloc_layout(sh), ep.alloc_notify(sh)
    d2 = {k: torch.empty_like(v) for k, v in d1.items()}
    ep.ep_layout_notify_dispatch(sh, x, idx_d, wt_d, lay2, nt2, ws, d2, status, sc)
    assert ep.ep_sync_status(status) == ep.EP_OK
    assert int(sc.item()) == 0
    check_layout_notify(lay2, nt2, lay_ref, nt_ref)
    for k in d1:
        a, b = d1[k], d2[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"{k} differs from the separate calls"
    del d1, d2, x
    torch.cuda.empty_cache()


def test_fused_stall_times_out_and_next_call_is_exact():
    """A layout + notify tile that never publishes makes the tiles after it
    give up (EP_ERR_TIMEOUT); dispatch still stays inside its buffers, the
    counter ends at zero, and the next call is bit-exact."""
    w = CASES["r24_many_tiles"]
    idx, wt = gen_routing(w)
    x = gen_x(w)
    lay_ref, nt_ref, dp = _oracle_all(w, idx, wt, x)
    sh, lay, nt, disp = _buffers(w)
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, dtype=torch.int64, device="cuda")
    ep.ep_debug_layout_notify_dispatch_stall(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status,
                                             stall_tile=1, wait_limit_us=2000, sched=sc)
    assert ep.ep_sync_status(status) == ep.EP_ERR_TIMEOUT
    assert int(sc.item()) == 0
    status.zero_()
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status, sc)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    _check_dispatch(disp, dp, int(nt_ref["recv_base"][-1]))


def test_fused_first_call_inside_graph_capture_and_shared_workspace():
    """First call of a new shape inside a CUDA-graph capture; replays on new
    inputs match the oracle; the same workspace serves ep_layout_notify calls
    in between."""
    w = Workload("e", R=16, T=200, H=512, E=128, K=6, C=5, mask=0.05)
    sh = shape_of(w)
    lay, nt, disp = ep.alloc_layout(sh), ep.alloc_notify(sh), ep.alloc_dispatch(sh, worst_case_rows(w))
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, dtype=torch.int64, device="cuda")
    x_d = torch.empty(w.R, w.T, w.H, dtype=torch.bfloat16, device="cuda")
    idx_d = torch.empty(w.R, w.T, w.K, dtype=torch.int64, device="cuda")
    wt_d = torch.empty(w.R, w.T, w.K, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ep.ep_layout_notify_dispatch(sh, x_d, idx_d, wt_d, lay, nt, ws, disp, status, sc, stream=stream)
    for seed in (3, 4):
        ws_ = w.replace(seed=seed)
        idx, wt = gen_routing(ws_)
        x = gen_x(ws_)
        idx_d.copy_(idx)
        wt_d.copy_(wt)
        x_d.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_sync_status(status) == ep.EP_OK
        lay_ref, nt_ref, dp = _oracle_all(ws_, idx, wt, x)
        check_layout_notify(lay, nt, lay_ref, nt_ref)
        _check_dispatch(disp, dp, int(nt_ref["recv_base"][-1]))
        # the workspace also serves an ep_layout_notify call in between
        lay2, nt2 = ep.alloc_layout(sh), ep.alloc_notify(sh)
        ep.ep_layout_notify(sh, idx_d, lay2, nt2, ws, status)
        assert ep.ep_sync_status(status) == ep.EP_OK
        check_layout_notify(lay2, nt2, lay_ref, nt_ref)
    assert int(sc.item()) == 0


def test_fused_capacity_overflow_reports_status():
    """A receive pool of half the rows: EP_ERR_CAPACITY, the rows that fit are
    exact, and the rows just past the pool are left untouched."""
    w = CASES["ragged_r16_zipf"]
    idx, wt = gen_routing(w)
    x = gen_x(w)
    lay_ref, nt_ref, dp = _oracle_all(w, idx, wt, x)
    cap = int(nt_ref["recv_base"][-1]) // 2
    sh, lay, nt, full = _buffers(w, cap=cap + 8)
    full["recv_x"].view(torch.int16).fill_(0x3C3C)
    disp = {k: v[:cap] for k, v in full.items()}
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status)
    assert ep.ep_sync_status(status) == ep.EP_ERR_CAPACITY
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    _check_dispatch(disp, {k: v[:cap] for k, v in dp.items()}, cap)
    assert bool((full["recv_x"][cap:].view(torch.int16) == 0x3C3C).all()), "rows past the pool were written"


def test_fused_bad_expert_id_reports_status():
    """Ids outside [-1, E): EP_ERR_INPUT; layout, notify and every dispatched
    row and field are those of the top-k with those slots empty."""
    w = CASES["r24_many_tiles"]
    idx, wt = gen_routing(w)
    x = gen_x(w)
    idx[7, 0, 2] = w.E
    idx[23, 1499, 5] = -9
    clean = idx.clone()
    clean[7, 0, 2] = -1
    clean[23, 1499, 5] = -1
    lay_ref, nt_ref, dp = _oracle_all(w, clean, wt, x)
    sh, lay, nt, disp = _buffers(w)
    ws = ep.alloc_layout_notify_workspace(sh)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_layout_notify_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), lay, nt, ws, disp, status)
    assert ep.ep_sync_status(status) == ep.EP_ERR_INPUT
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    _check_dispatch(disp, dp, int(nt_ref["recv_base"][-1]))
