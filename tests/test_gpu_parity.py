"""CUDA path vs the CPU oracle, element by element, through the C ABI.

* small workloads (tiny, low_latency, prefill) and edge shapes: every output
  of every step compared with the oracle (integers and bytes bit-exact,
  combine within |d| <= 1e-2 + 8e-3|ref| and bit-exact);
* full-size workloads (skewed, large): layout, notify and all dispatch
  metadata compared in full; the dispatched payload checked at full size by
  the property recv_x[p] == x[src_info[p]] plus oracle rows on a sample;
  combine checked at full size by the identity-expert closed form and, for
  random expert outputs, against the oracle on a sample of tokens.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import CONFIGS, Workload, worst_case_rows
from gpu_util import (assert_combine_close, assert_equal, check_layout_notify, make_inputs,
                      run_layout_notify, shape_of, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.lib()


def full_parity(w: Workload, random_expert: bool = True, capacity: int | None = None):
    """Run all four steps and compare every output with the oracle."""
    o = oracle.load()
    idx, wt, x = make_inputs(w)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    lay, nt, dp, cb = oracle.run_all(w.R, w.T, w.K, w.E, w.H, w.C, w.expert_alignment, xb,
                                     idx.numpy(), wt.numpy(), o)
    rows = int(nt["recv_base"][-1])
    sh = shape_of(w)
    pipe = ep.Pipeline(sh, capacity if capacity is not None else max(1, worst_case_rows(w)))
    cx, cw = pipe.run(x.cuda(), idx.cuda(), wt.cuda())
    assert ep.ep_sync_status(pipe.status) == ep.EP_OK
    check_layout_notify(pipe.layout, pipe.notify, lay, nt)
    D = pipe.dispatch
    assert_equal("recv_x", u16(D["recv_x"][:rows]), dp["recv_x"])
    assert_equal("recv_topk_idx", D["recv_topk_idx"][:rows].cpu().numpy(), dp["recv_topk_idx"])
    assert_equal("recv_topk_w", D["recv_topk_w"][:rows].cpu().numpy(), dp["recv_topk_w"])
    assert_equal("recv_src_info", D["recv_src_info"][:rows].cpu().numpy(), dp["recv_src_info"])
    assert_combine_close("combined_x", u16(cx), cb["combined_x"])
    assert_equal("combined_w", cw.cpu().numpy(), cb["combined_w"])

    # a second run gives byte-identical results
    snap = {k: v.clone() for k, v in pipe.notify.items() if k != "workspace"}
    snap_cx = cx.clone()
    pipe.run(x.cuda(), idx.cuda(), wt.cuda())
    assert ep.ep_sync_status(pipe.status) == ep.EP_OK
    for k, v in snap.items():
        assert torch.equal(v, pipe.notify[k]), f"{k} differs between runs"
    assert torch.equal(snap_cx.view(torch.int16), cx.view(torch.int16))

    if random_expert and rows > 0:
        # an expert whose outputs differ per row: order of the sum matters
        g = torch.Generator().manual_seed(1234)
        y = (torch.randn(rows, w.H, generator=g) * 3).to(torch.bfloat16)
        yw = torch.randn(rows, w.K, generator=g)
        ref = o.combine(w.R, w.T, w.K, w.H, y.view(torch.int16).numpy().view(np.uint16), yw.numpy(),
                        nt["send_pos"], nt["recv_base"])
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = ep.alloc_combine(sh)
        ep.ep_combine(sh, y.cuda(), yw.cuda(), pipe.notify["send_pos"], pipe.notify["recv_base"],
                      out["combined_x"], out["combined_w"], status)
        assert ep.ep_sync_status(status) == ep.EP_OK
        assert_combine_close("combined_x (random expert)", u16(out["combined_x"]), ref["combined_x"])
        assert_equal("combined_w (random expert)", out["combined_w"].cpu().numpy(), ref["combined_w"])
    return pipe


@pytest.mark.parametrize("name", ["tiny", "low_latency", "prefill"])
def test_workload_full_parity(name):
    full_parity(CONFIGS[name])


EDGE = {
    "single_rank": Workload("e", R=1, T=37, H=64, E=6, K=3, C=4, routing="replace", mask=0.2),
    "empty_tokens": Workload("e", R=4, T=0, H=64, E=8, K=2, C=3),
    "channels_exceed_tokens": Workload("e", R=8, T=50, H=128, E=64, K=4, C=64, mask=0.1),
    "top1_counting_sort": Workload("e", R=16, T=33, H=256, E=64, K=1, C=5),
    "r32_min_hidden_repeats": Workload("e", R=32, T=19, H=8, E=256, K=8, C=3, routing="replace",
                                       mask=0.3),
    "all_masked": Workload("e", R=8, T=40, H=64, E=16, K=4, C=4, mask=1.0),
    "ragged_hidden": Workload("e", R=4, T=70, H=264, E=8, K=3, C=7, routing="zipf"),
    "odd_ranks_align": Workload("e", R=3, T=41, H=72, E=9, K=2, C=5, expert_alignment=4),
    "align128": Workload("e", R=16, T=64, H=512, E=128, K=8, C=6, expert_alignment=128),
    "odd_topk": Workload("e", R=8, T=29, H=1024, E=32, K=5, C=2, mask=0.15),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_parity(case):
    full_parity(EDGE[case])


def _sample_tokens(R, T, n, seed):
    rng = np.random.default_rng(seed)
    g = rng.choice(R * T, size=min(n, R * T), replace=False)
    return np.sort(g)


@pytest.mark.parametrize("name", ["skewed", "large"])
def test_workload_full_size(name):
    """Full-size layout/notify/metadata parity, payload property + sampled rows,
    combine closed form + sampled oracle tokens."""
    w = CONFIGS[name]
    o = oracle.load()
    idx, wt, x = make_inputs(w, x_on_gpu=True)
    lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
    rows = int(nt_ref["recv_base"][-1])
    sh = shape_of(w)
    pipe = ep.Pipeline(sh, rows)
    cx, cw = pipe.run(x, idx.cuda(), wt.cuda())
    assert ep.ep_sync_status(pipe.status) == ep.EP_OK
    check_layout_notify(pipe.layout, pipe.notify, lay_ref, nt_ref)

    # dispatch metadata in full
    dp_ref = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, None, idx.numpy(), wt.numpy(),
                        nt_ref["send_pos"], nt_ref["recv_base"], payload=False)
    D = pipe.dispatch
    src = D["recv_src_info"].cpu().numpy()
    assert_equal("recv_src_info", src, dp_ref["recv_src_info"])
    assert_equal("recv_topk_idx", D["recv_topk_idx"].cpu().numpy(), dp_ref["recv_topk_idx"])
    assert_equal("recv_topk_w", D["recv_topk_w"].cpu().numpy(), dp_ref["recv_topk_w"])

    # payload: every row is a bit copy of its source row (full size, on device)
    xf = x.view(torch.int16).view(-1, w.H)
    src_g = torch.from_numpy(src[:, 0].astype(np.int64) * w.T + src[:, 1]).cuda()
    rx = D["recv_x"].view(torch.int16)
    for a in range(0, rows, 1 << 18):
        b = min(rows, a + (1 << 18))
        assert torch.equal(rx[a:b], xf[src_g[a:b]]), f"recv_x rows {a}..{b} differ from their source"
    # payload: oracle dispatch of a sample of rows
    pick = np.random.default_rng(5).choice(rows, size=min(rows, 2000), replace=False)
    want = xf[src_g[torch.from_numpy(pick).cuda()]].cpu().numpy().view(np.uint16)
    assert_equal("recv_x sample", rx[torch.from_numpy(pick).cuda()].cpu().numpy().view(np.uint16), want)

    # combine, identity expert, full size: bf16(n_dest * x); +0 without destination
    n_dest = (pipe.notify["send_pos"] >= 0).sum(-1).view(-1)
    cxf = cx.view(-1, w.H)
    for a in range(0, w.R * w.T, 1 << 16):
        b = min(w.R * w.T, a + (1 << 16))
        n = n_dest[a:b].to(torch.float32)[:, None]
        exp = (x.view(-1, w.H)[a:b].float() * n).to(torch.bfloat16)
        exp = torch.where(n == 0, torch.zeros_like(exp), exp)
        assert torch.equal(cxf[a:b].view(torch.int16), exp.view(torch.int16)), f"combined rows {a}..{b}"
    tw = wt.cuda()
    assert torch.equal(cw, torch.where(idx.cuda() >= 0, tw, torch.zeros_like(tw))), "combined_w"

    # combine, random expert outputs, oracle on sampled tokens
    gen = torch.Generator(device="cuda").manual_seed(77)
    for a in range(0, rows, 1 << 16):
        b = min(rows, a + (1 << 16))
        D["recv_x"][a:b].copy_(torch.randn(b - a, w.H, generator=gen, device="cuda").mul_(3))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_combine(sh, D["recv_x"], D["recv_topk_w"], pipe.notify["send_pos"], pipe.notify["recv_base"],
                  cx, cw, status)
    assert ep.ep_sync_status(status) == ep.EP_OK
    toks = _sample_tokens(w.R, w.T, 1024, 9)
    sp = nt_ref["send_pos"].reshape(-1, w.R)[toks]          # [n, R]
    base = nt_ref["recv_base"]
    rows_needed = [int(base[r] + sp[i, r]) for i in range(len(toks)) for r in range(w.R) if sp[i, r] >= 0]
    y_small = D["recv_x"][torch.tensor(rows_needed, device="cuda")].view(torch.int16).cpu().numpy().view(np.uint16)
    yw_small = D["recv_topk_w"][torch.tensor(rows_needed, device="cuda")].cpu().numpy()
    # sub-problem: the sampled tokens as source rank 0, their rows numbered 0.. in order
    sub_sp = -np.ones((w.R, len(toks), w.R), np.int32)
    k = 0
    for i in range(len(toks)):
        for r in range(w.R):
            if sp[i, r] >= 0:
                sub_sp[0, i, r] = k
                k += 1
    ref = o.combine(w.R, len(toks), w.K, w.H, y_small, yw_small, sub_sp, np.zeros(w.R + 1, np.int64))
    got = cx.view(-1, w.H)[torch.from_numpy(toks).cuda()]
    assert_combine_close("combined_x sample (random expert)", u16(got), ref["combined_x"][0])
    assert_equal("combined_w sample", cw.view(-1, w.K)[torch.from_numpy(toks).cuda()].cpu().numpy(),
                 ref["combined_w"][0])


# ---------------------------------------------------------------------------- errors
def test_capacity_overflow_reports_status():
    w = CONFIGS["tiny"]
    idx, wt, x = make_inputs(w)
    o = oracle.load()
    xb = x.view(torch.int16).numpy().view(np.uint16)
    lay, nt, dp, cb = oracle.run_all(w.R, w.T, w.K, w.E, w.H, w.C, 1, xb, idx.numpy(), wt.numpy(), o)
    rows = int(nt["recv_base"][-1])
    cap = rows // 2
    pipe = ep.Pipeline(shape_of(w), cap)
    pipe.run(x.cuda(), idx.cuda(), wt.cuda())
    assert ep.ep_sync_status(pipe.status) == ep.EP_ERR_CAPACITY
    # rows that fit are still exact
    assert_equal("recv_x within capacity", u16(pipe.dispatch["recv_x"]), dp["recv_x"][:cap])
    assert_equal("recv_src_info within capacity", pipe.dispatch["recv_src_info"].cpu().numpy(),
                 dp["recv_src_info"][:cap])


def test_bad_expert_id_reports_status():
    w = CONFIGS["tiny"]
    idx, wt, x = make_inputs(w)
    idx = idx.clone()
    idx[1, 5, 0] = w.E + 3
    sh, lay, nt, status = run_layout_notify(w, idx)
    assert ep.ep_sync_status(status) == ep.EP_ERR_INPUT


def test_inconsistent_counts_report_status():
    w = CONFIGS["low_latency"]
    idx, wt, x = make_inputs(w)
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    lay["num_tokens_per_rank"][3, 5] += 1
    ep.ep_notify_dispatch(sh, lay["is_token_in_rank"], lay["num_tokens_per_rank"],
                          lay["num_tokens_per_rdma_rank"], lay["num_tokens_per_expert"], nt,
                          nt["workspace"], status)
    assert ep.ep_sync_status(status) == ep.EP_ERR_INCONSISTENT


def test_stalled_lookback_times_out_and_context_survives():
    """A block that never publishes: waiting blocks give up after the limit,
    report EP_ERR_TIMEOUT, and the next normal run is correct."""
    w = CONFIGS["low_latency"]
    idx, wt, x = make_inputs(w)
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    ep.ep_debug_notify_dispatch_stall(sh, lay["is_token_in_rank"], lay["num_tokens_per_rank"],
                                      lay["num_tokens_per_rdma_rank"], lay["num_tokens_per_expert"], nt,
                                      nt["workspace"], status, stall_block=5, wait_limit_us=2000)
    assert ep.ep_sync_status(status) == ep.EP_ERR_TIMEOUT
    # the context is still usable: a normal run matches the oracle
    full_parity(CONFIGS["tiny"], random_expert=False)


@pytest.mark.parametrize("dynamic", [False, True], ids=["static", "dynamic"])
def test_stalled_dispatch_times_out_and_context_survives(dynamic):
    """A dispatch CTA whose storer never frees a ring slot: its producer's and
    storer's bounded waits run out, the status word reports EP_ERR_TIMEOUT, the
    other CTAs finish, and the next normal dispatch on the same buffers is
    bit-exact."""
    # 4 KB rows: 36 units for CTA 0 against a 16-slot ring, so its producer
    # has to wait for a free slot
    w = Workload("e", R=8, T=2048, H=2048, E=64, K=4, C=4)
    idx, wt, x = make_inputs(w)
    sh = shape_of(w)
    o = oracle.load()
    lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
    rows = int(nt_ref["recv_base"][-1])
    sp, rb = torch.from_numpy(nt_ref["send_pos"]).cuda(), torch.from_numpy(nt_ref["recv_base"]).cuda()
    D = ep.alloc_dispatch(sh, rows)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sched = torch.zeros(1, dtype=torch.int64, device="cuda") if dynamic else None
    ep.ep_debug_dispatch_stall(sh, x.cuda(), idx.cuda(), wt.cuda(), sp, rb, D["recv_x"], D["recv_topk_idx"],
                               D["recv_topk_w"], D["recv_src_info"], status, stall_cta=0, wait_limit_us=2000,
                               sched=sched)
    assert ep.ep_sync_status(status) == ep.EP_ERR_TIMEOUT
    if dynamic:  # the stalled CTA took the rest of the units and the counter still ended at zero
        assert int(sched.item()) == 0
    status.zero_()
    ep.ep_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), sp, rb, D["recv_x"], D["recv_topk_idx"], D["recv_topk_w"],
                   D["recv_src_info"], status, sched=sched)
    assert ep.ep_sync_status(status) == ep.EP_OK
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x.view(torch.int16).numpy().view(np.uint16), idx.numpy(),
                    wt.numpy(), nt_ref["send_pos"], nt_ref["recv_base"])
    assert_equal("recv_x after a stalled run", u16(D["recv_x"]), dp["recv_x"])
    assert_equal("recv_src_info after a stalled run", D["recv_src_info"].cpu().numpy(), dp["recv_src_info"])


@pytest.mark.parametrize("name", ["prefill_like", "fp8_rows_like", "tiny"])
def test_dispatch_dynamic_assignment_matches_oracle(name):
    """Row parts handed out through the sched counter: bit-exact, whatever CTA
    takes which unit, and the counter is back at zero after every call."""
    w = {"prefill_like": Workload("e", R=8, T=1024, H=7168, E=64, K=8, C=6),
         "fp8_rows_like": Workload("e", R=16, T=512, H=2048, E=128, K=6, C=4, routing="zipf"),
         "tiny": CONFIGS["tiny"]}[name]
    idx, wt, x = make_inputs(w)
    o = oracle.load()
    lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x.view(torch.int16).numpy().view(np.uint16), idx.numpy(),
                    wt.numpy(), nt_ref["send_pos"], nt_ref["recv_base"])
    rows = int(nt_ref["recv_base"][-1])
    sh = shape_of(w)
    sp, rb = torch.from_numpy(nt_ref["send_pos"]).cuda(), torch.from_numpy(nt_ref["recv_base"]).cuda()
    sched = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        D = ep.alloc_dispatch(sh, max(rows, 1))
        ep.ep_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), sp, rb, D["recv_x"], D["recv_topk_idx"],
                       D["recv_topk_w"], D["recv_src_info"], status, sched=sched)
        assert ep.ep_sync_status(status) == ep.EP_OK
        assert int(sched.item()) == 0
        assert_equal("recv_x (dynamic)", u16(D["recv_x"][:rows]), dp["recv_x"])
        assert_equal("recv_topk_idx (dynamic)", D["recv_topk_idx"][:rows].cpu().numpy(), dp["recv_topk_idx"])
        assert_equal("recv_topk_w (dynamic)", D["recv_topk_w"][:rows].cpu().numpy(), dp["recv_topk_w"])
        assert_equal("recv_src_info (dynamic)", D["recv_src_info"][:rows].cpu().numpy(), dp["recv_src_info"])


def test_dispatch_concurrent_streams_with_own_sched_words():
    """Two dispatch calls running at the same time on two streams, each with its
    own sched word: both bit-exact, both words back at zero."""
    w = Workload("e", R=8, T=1024, H=4096, E=64, K=8, C=6)
    o = oracle.load()
    sh = shape_of(w)
    runs = []
    for seed in (21, 22):
        ws = Workload(w.name, R=w.R, T=w.T, H=w.H, E=w.E, K=w.K, C=w.C, seed=seed)
        idx, wt, x = make_inputs(ws)
        lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
        nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
        rows = int(nt_ref["recv_base"][-1])
        dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x.view(torch.int16).numpy().view(np.uint16), idx.numpy(),
                        wt.numpy(), nt_ref["send_pos"], nt_ref["recv_base"])
        dev = dict(x=x.cuda(), idx=idx.cuda(), wt=wt.cuda(), sp=torch.from_numpy(nt_ref["send_pos"]).cuda(),
                   rb=torch.from_numpy(nt_ref["recv_base"]).cuda(), D=ep.alloc_dispatch(sh, rows),
                   st=torch.zeros(1, dtype=torch.int32, device="cuda"),
                   sched=torch.zeros(1, dtype=torch.int64, device="cuda"), stream=torch.cuda.Stream())
        runs.append((dev, dp, rows))
    torch.cuda.synchronize()
    for _ in range(3):
        for dev, _, _ in runs:
            D = dev["D"]
            ep.ep_dispatch(sh, dev["x"], dev["idx"], dev["wt"], dev["sp"], dev["rb"], D["recv_x"], D["recv_topk_idx"],
                           D["recv_topk_w"], D["recv_src_info"], dev["st"], stream=dev["stream"], sched=dev["sched"])
    torch.cuda.synchronize()
    for dev, dp, rows in runs:
        assert ep.ep_sync_status(dev["st"]) == ep.EP_OK
        assert int(dev["sched"].item()) == 0
        assert_equal("recv_x (concurrent)", u16(dev["D"]["recv_x"][:rows]), dp["recv_x"])
        assert_equal("recv_src_info (concurrent)", dev["D"]["recv_src_info"][:rows].cpu().numpy(), dp["recv_src_info"])


def test_sched_word_stays_consistent_over_a_mixed_sequence():
    """One sched word shared by a long sequence of calls of different shapes and
    kinds (bf16, FP8, low-latency layout; small calls that keep the static split,
    large ones that use the counter; calls that time out on purpose): it reads
    zero after every call, and a final call is bit-exact."""
    o = oracle.load()
    sched = torch.zeros(1, dtype=torch.int64, device="cuda")
    rng = np.random.default_rng(11)
    shapes = [Workload("e", R=8, T=1024, H=4096, E=64, K=8, C=4), Workload("e", R=16, T=64, H=512, E=32, K=4, C=2),
              Workload("e", R=4, T=2048, H=1024, E=16, K=2, C=3, routing="zipf")]
    prepared = []
    for w in shapes:
        idx, wt, x = make_inputs(w)
        lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
        nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
        rows = int(nt_ref["recv_base"][-1])
        prepared.append((w, idx, wt, x, nt_ref, rows))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(40):
        w, idx, wt, x, nt_ref, rows = prepared[int(rng.integers(len(prepared)))]
        sh = shape_of(w)
        sp, rb = torch.from_numpy(nt_ref["send_pos"]).cuda(), torch.from_numpy(nt_ref["recv_base"]).cuda()
        D = ep.alloc_dispatch(sh, rows)
        kind = int(rng.integers(4))
        status.zero_()
        if kind == 0:
            ep.ep_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), sp, rb, D["recv_x"], D["recv_topk_idx"],
                           D["recv_topk_w"], D["recv_src_info"], status, sched=sched)
            assert ep.ep_sync_status(status) == ep.EP_OK
        elif kind == 1:
            x8 = torch.randint(0, 256, (w.R, w.T, w.H), dtype=torch.uint8, device="cuda")
            r8 = torch.empty(rows, w.H, dtype=torch.uint8, device="cuda")
            ep.ep_dispatch_fp8(sh, x8, None, idx.cuda(), wt.cuda(), sp, rb, r8, None, D["recv_topk_idx"],
                               D["recv_topk_w"], D["recv_src_info"], status, sched=sched)
            assert ep.ep_sync_status(status) == ep.EP_OK
        elif kind == 2:
            cap = w.R * w.T
            slot = torch.empty(w.R, w.T, w.K, dtype=torch.int32, device="cuda")
            ep.ep_ll_layout(sh, idx.cuda(), None, cap, slot, torch.empty(w.E, w.R, 2, dtype=torch.int32, device="cuda"),
                            torch.empty(w.E, dtype=torch.int32, device="cuda"), status)
            rx = torch.empty(w.E, cap, w.H, dtype=torch.bfloat16, device="cuda")
            ep.ep_ll_dispatch(sh, x.cuda(), idx.cuda(), slot, cap, rx, None, status, sched=sched)
            assert ep.ep_sync_status(status) == ep.EP_OK
        else:
            ep.ep_debug_dispatch_stall(sh, x.cuda(), idx.cuda(), wt.cuda(), sp, rb, D["recv_x"], D["recv_topk_idx"],
                                       D["recv_topk_w"], D["recv_src_info"], status, stall_cta=1,
                                       wait_limit_us=1000, sched=sched)
            assert ep.ep_sync_status(status) in (ep.EP_OK, ep.EP_ERR_TIMEOUT)
        assert int(sched.item()) == 0, f"sched not zero after call {step} (kind {kind})"
    w, idx, wt, x, nt_ref, rows = prepared[0]
    sh = shape_of(w)
    D = ep.alloc_dispatch(sh, rows)
    status.zero_()
    ep.ep_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), torch.from_numpy(nt_ref["send_pos"]).cuda(),
                   torch.from_numpy(nt_ref["recv_base"]).cuda(), D["recv_x"], D["recv_topk_idx"], D["recv_topk_w"],
                   D["recv_src_info"], status, sched=sched)
    assert ep.ep_sync_status(status) == ep.EP_OK
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x.view(torch.int16).numpy().view(np.uint16), idx.numpy(),
                    wt.numpy(), nt_ref["send_pos"], nt_ref["recv_base"])
    assert_equal("recv_x after the sequence", u16(D["recv_x"][:rows]), dp["recv_x"])


def test_invalid_arguments_rejected_on_host():
    w = CONFIGS["tiny"]
    idx, wt, x = make_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = ep.EpShape.make(12, 16, 2, 24, 256, 2)  # 12 ranks: not whole nodes
    lay = ep.alloc_layout(ep.EpShape.make(2, 16, 2, 24, 256, 2))
    rc = ep.lib().ep_get_dispatch_layout(
        __import__("ctypes").byref(bad), ep._vp(idx.cuda().data_ptr()),
        ep._vp(lay["num_tokens_per_rank"].data_ptr()), ep._vp(lay["num_tokens_per_rdma_rank"].data_ptr()),
        ep._vp(lay["num_tokens_per_expert"].data_ptr()), ep._vp(lay["is_token_in_rank"].data_ptr()),
        ep._vp(status.data_ptr()), ep._vp(0))
    assert rc == ep.EP_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        ep.ep_get_dispatch_layout(shape_of(w), idx, *[None] * 4, status)  # CPU tensor
    with pytest.raises(ep.EpError):
        sh = shape_of(w)
        misaligned = torch.empty(w.R * w.T * w.K + 1, dtype=torch.int64, device="cuda")[1:].view(w.R, w.T, w.K)
        L = ep.alloc_layout(sh)
        ep.ep_get_dispatch_layout(sh, misaligned, L["num_tokens_per_rank"], L["num_tokens_per_rdma_rank"],
                                  L["num_tokens_per_expert"], L["is_token_in_rank"], status)


def test_host_mapped_receive_counts():
    """notify can publish the receive counts into host-mapped pinned memory."""
    w = CONFIGS["low_latency"]
    idx, wt, x = make_inputs(w)
    o = oracle.load()
    nt_ref = o.notify(w.R, w.T, w.E, w.C, 1, o.layout(w.R, w.T, w.K, w.E, idx.numpy()))
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    host = torch.full((w.R + 1,), -1, dtype=torch.int32).pin_memory()
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    ep.ep_notify_dispatch(sh, lay["is_token_in_rank"], lay["num_tokens_per_rank"],
                          lay["num_tokens_per_rdma_rank"], lay["num_tokens_per_expert"], nt,
                          nt["workspace"], status, host_num_recv_tokens=host)
    assert ep.ep_sync_status(status) == ep.EP_OK
    want = np.concatenate([nt_ref["num_recv_tokens"], [nt_ref["recv_base"][-1]]]).astype(np.int32)
    assert_equal("host_num_recv_tokens", host.numpy(), want)


def test_workspace_reused_across_shapes_and_after_a_timeout():
    """One notify workspace, zeroed once, serves calls of different shapes in
    turn and stays valid after a call whose waits ran out."""
    o = oracle.load()
    shapes = [CONFIGS["low_latency"], CONFIGS["tiny"], EDGE["r32_min_hidden_repeats"], CONFIGS["low_latency"]]
    biggest = max(ep.ep_notify_workspace_bytes(shape_of(w)) for w in shapes)
    ws = torch.zeros(biggest, dtype=torch.uint8, device="cuda")
    for i, w in enumerate(shapes):
        idx, wt, x = make_inputs(w)
        sh = shape_of(w)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        lay = ep.alloc_layout(sh)
        nt = ep.alloc_notify(sh)
        ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                                  lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
        args = (lay["is_token_in_rank"], lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                lay["num_tokens_per_expert"], nt)
        if i == 1:  # a call that times out in the middle of the sequence
            ep.ep_debug_notify_dispatch_stall(sh, *args, ws, status, stall_block=0, wait_limit_us=2000)
            assert ep.ep_sync_status(status) == ep.EP_ERR_TIMEOUT
            status.zero_()
        ep.ep_notify_dispatch(sh, *args, ws, status)
        assert ep.ep_sync_status(status) == ep.EP_OK
        lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
        check_layout_notify(lay, nt, lay_ref, o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref))


@pytest.mark.parametrize("name", ["tiny", "low_latency", "prefill", "channels_exceed_tokens", "odd_ranks_align",
                                  "r32_min_hidden_repeats", "empty_tokens"])
def test_notify_lookback_path_matches_oracle(name):
    """Small sources normally take notify's recount path; the test hook forces
    the inter-block lookback path on the same shapes, which must agree too."""
    w = CONFIGS.get(name) or EDGE[name]
    o = oracle.load()
    idx, wt, x = make_inputs(w)
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    for _ in range(2):  # twice: the second call reuses the workspace state of the first
        ep.ep_debug_notify_dispatch_stall(sh, lay["is_token_in_rank"], lay["num_tokens_per_rank"],
                                          lay["num_tokens_per_rdma_rank"], lay["num_tokens_per_expert"], nt,
                                          nt["workspace"], status, stall_block=-1, wait_limit_us=1000000)
        assert ep.ep_sync_status(status) == ep.EP_OK
        lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
        check_layout_notify(lay, nt, lay_ref, o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref))



@pytest.mark.parametrize("name", ["low_latency", "r32_min_hidden_repeats", "all_masked"])
def test_cached_mode_reuses_the_handle(name):
    """Cached mode: a handle from one full step serves a later step with the same
    routing and new activations; only rows move, combine matches the oracle."""
    w = CONFIGS.get(name) or EDGE[name]
    o = oracle.load()
    idx, wt, x1 = make_inputs(w)
    x2 = gen_x_seeded(w, 99)
    pipe = ep.Pipeline(shape_of(w), max(1, worst_case_rows(w)))
    pipe.run(x1.cuda(), idx.cuda(), wt.cuda())
    assert ep.ep_sync_status(pipe.status) == ep.EP_OK
    src_before = pipe.dispatch["recv_src_info"].clone()
    cx = pipe.run_cached(x2.cuda())
    assert ep.ep_sync_status(pipe.status) == ep.EP_OK
    xb = x2.view(torch.int16).numpy().view(np.uint16)
    lay = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay)
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, xb, idx.numpy(), wt.numpy(), nt["send_pos"], nt["recv_base"],
                    with_topk=False)
    rows = int(nt["recv_base"][-1])
    assert_equal("recv_x (cached)", u16(pipe.dispatch["recv_x"][:rows]), dp["recv_x"])
    assert torch.equal(src_before, pipe.dispatch["recv_src_info"])  # not rewritten
    cb = o.combine(w.R, w.T, w.K, w.H, dp["recv_x"], None, nt["send_pos"], nt["recv_base"])
    assert_combine_close("combined_x (cached)", u16(cx), cb["combined_x"])


def gen_x_seeded(w, seed):
    from combine_get_dispatch_notify_gb300.workloads import gen_x
    return gen_x(w.replace(seed=seed))


@pytest.mark.parametrize("name", ["tiny", "low_latency", "prefill", "top1_counting_sort", "channels_exceed_tokens"])
@pytest.mark.parametrize("cached", [False, True], ids=["full", "cached"])
def test_dispatch_fp8_matches_oracle(name, cached):
    """FP8 rows (bytes) and their per-token scales go where the bf16 rows go."""
    w = CONFIGS.get(name) or EDGE[name]
    o = oracle.load()
    idx, wt, _ = make_inputs(w)
    g = torch.Generator().manual_seed(5)
    S = max(1, w.H // 128)
    xb = torch.randint(0, 256, (w.R, w.T, w.H), generator=g, dtype=torch.uint8)
    xs = torch.randn(w.R, w.T, S, generator=g)
    sh, lay, nt, status = run_layout_notify(w, idx)
    cap = max(1, worst_case_rows(w))
    rx = torch.empty(cap, w.H, dtype=torch.uint8, device="cuda")
    rs = torch.empty(cap, S, dtype=torch.float32, device="cuda")
    rti = None if cached else torch.empty(cap, w.K, dtype=torch.int64, device="cuda")
    rtw = None if cached else torch.empty(cap, w.K, dtype=torch.float32, device="cuda")
    rsi = torch.empty(cap, 2, dtype=torch.int32, device="cuda")
    sched = None if cached else torch.zeros(1, dtype=torch.int64, device="cuda")  # dynamic / static split
    ep.ep_dispatch_fp8(sh, xb.cuda(), xs.cuda(), None if cached else idx.cuda(), None if cached else wt.cuda(),
                       nt["send_pos"], nt["recv_base"], rx, rs, rti, rtw, rsi, status, sched=sched)
    assert ep.ep_sync_status(status) == ep.EP_OK
    assert sched is None or int(sched.item()) == 0
    lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
    ref = o.dispatch_fp8(w.R, w.T, w.K, w.E, w.H, w.C, xb.numpy(), xs.numpy(), idx.numpy(), wt.numpy(),
                         nt_ref["send_pos"], nt_ref["recv_base"], with_topk=not cached)
    rows = int(nt_ref["recv_base"][-1])
    assert_equal("recv_x (fp8)", rx[:rows].cpu().numpy(), ref["recv_x"])
    assert_equal("recv_x_scales", rs[:rows].cpu().numpy(), ref["recv_x_scales"])
    assert_equal("recv_src_info", rsi[:rows].cpu().numpy(), ref["recv_src_info"])
    if not cached:
        assert_equal("recv_topk_idx", rti[:rows].cpu().numpy(), ref["recv_topk_idx"])
        assert_equal("recv_topk_w", rtw[:rows].cpu().numpy(), ref["recv_topk_w"])


# ---------------------------------------------------------------------------- low-latency layout
LL_CASES = {
    "tiny": (CONFIGS["tiny"], 1),
    # enough row parts per CTA that ll_dispatch takes units from the sched counter
    "counter_sized": (Workload("e", R=8, T=2048, H=2048, E=64, K=8, C=4), 1),
    "low_latency": (CONFIGS["low_latency"], 1),
    "top1_counting_sort": (EDGE["top1_counting_sort"], 1),
    "r32_min_hidden_repeats": (EDGE["r32_min_hidden_repeats"], None),  # repeated experts: cap R*T*K
    "all_masked": (EDGE["all_masked"], 1),
    "odd_ranks_align": (EDGE["odd_ranks_align"], 1),
}


def _ll_run(w, cap, idx, wt, x, y=None):
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    slot = torch.empty(w.R, w.T, w.K, dtype=torch.int32, device="cuda")
    rng_ = torch.empty(w.E, w.R, 2, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.E, dtype=torch.int32, device="cuda")
    ep.ep_ll_layout(sh, idx.cuda(), lay["num_tokens_per_expert"], cap, slot, rng_, cnt, status)
    rx = torch.zeros(w.E, cap, w.H, dtype=torch.bfloat16, device="cuda")
    src = torch.full((w.E, cap, 2), -1, dtype=torch.int32, device="cuda")
    sched = torch.zeros(1, dtype=torch.int64, device="cuda")
    ep.ep_ll_dispatch(sh, x, idx.cuda(), slot, cap, rx, src, status, sched=sched)
    out = torch.empty(w.R, w.T, w.H, dtype=torch.bfloat16, device="cuda")
    ep.ep_ll_combine(sh, rx if y is None else y, cap, idx.cuda(), wt.cuda(), slot, out, status)
    return status, slot, rng_, cnt, rx, src, out


@pytest.mark.parametrize("name", sorted(LL_CASES))
def test_ll_layout_dispatch_combine(name):
    w, capf = LL_CASES[name]
    cap = w.R * w.T * (capf or w.K)
    o = oracle.load()
    idx, wt, x = make_inputs(w)
    status, slot, rng_, cnt, rx, src, out = _ll_run(w, cap, idx, wt, x.cuda())
    assert ep.ep_sync_status(status) == ep.EP_OK
    ref = oracle.ll_layout(o, w.R, w.T, w.K, w.E, cap, idx.numpy())
    assert_equal("ll slot_pos", slot.cpu().numpy(), ref["slot_pos"])
    assert_equal("ll layout_range", rng_.cpu().numpy(), ref["layout_range"])
    assert_equal("ll count", cnt.cpu().numpy(), ref["count"])
    # every slot's row holds its token and source info (all slots, any size)
    s_i, t_i, k_i = np.nonzero(idx.numpy() >= 0)
    e_i = idx.numpy()[s_i, t_i, k_i]
    p_i = ref["slot_pos"][s_i, t_i, k_i]
    if len(s_i):
        ei, pi = torch.from_numpy(e_i).cuda(), torch.from_numpy(p_i.astype(np.int64)).cuda()
        got = rx[ei, pi].view(torch.int16)
        want = x.cuda().view(torch.int16)[torch.from_numpy(s_i).cuda(), torch.from_numpy(t_i).cuda()]
        assert torch.equal(got, want), "ll recv_x rows differ from their tokens"
        assert_equal("ll recv_src_info", src[ei, pi].cpu().numpy(), np.stack([s_i, t_i], 1).astype(np.int32))
    assert int((src[..., 0] >= 0).sum()) == len(s_i)  # nothing else written
    # combine: oracle on the whole problem when it is small, else on sampled tokens
    rows_bytes = w.E * cap * w.H * 2
    if rows_bytes <= (1 << 30):
        refc = oracle.ll_combine(o, w.R, w.T, w.K, w.E, w.H, cap, u16(rx), idx.numpy(), wt.numpy(),
                                 ref["slot_pos"])
        assert_combine_close("ll combined_x", u16(out), refc)
    else:
        toks = _sample_tokens(w.R, w.T, 256, 3)
        ti = idx.numpy().reshape(-1, w.K)[toks]
        sp = ref["slot_pos"].reshape(-1, w.K)[toks]
        n = len(toks)
        # sub-problem: one expert buffer holding row i*K + k for sampled token i, slot k
        rows = torch.zeros(n * w.K, w.H, dtype=torch.bfloat16, device="cuda")
        for i in range(n):
            for k in range(w.K):
                if ti[i, k] >= 0:
                    rows[i * w.K + k] = rx[int(ti[i, k]), int(sp[i, k])]
        sub_idx = np.where(ti >= 0, 0, -1).astype(np.int64).reshape(1, n, w.K)
        sub_pos = np.where(ti >= 0, np.arange(n * w.K).reshape(n, w.K), -1).astype(np.int32).reshape(1, n, w.K)
        refc = oracle.ll_combine(o, 1, n, w.K, 1, w.H, n * w.K, u16(rows), sub_idx,
                                 wt.numpy().reshape(-1, w.K)[toks].reshape(1, n, w.K), sub_pos)
        got = out.view(-1, w.H)[torch.from_numpy(toks).cuda()]
        assert_combine_close("ll combined_x (sampled)", u16(got), refc[0])


def test_ll_capacity_drop_reports_status():
    w = CONFIGS["tiny"]
    cap = 7  # far fewer rows than slots per expert
    o = oracle.load()
    idx, wt, x = make_inputs(w)
    status, slot, rng_, cnt, rx, src, out = _ll_run(w, cap, idx, wt, x.cuda())
    assert ep.ep_sync_status(status) == ep.EP_ERR_CAPACITY
    ref = oracle.ll_layout(o, w.R, w.T, w.K, w.E, cap, idx.numpy())
    assert ref["dropped"]
    assert_equal("ll slot_pos (capacity)", slot.cpu().numpy(), ref["slot_pos"])
    refc = oracle.ll_combine(o, w.R, w.T, w.K, w.E, w.H, cap, u16(rx), idx.numpy(), wt.numpy(), ref["slot_pos"])
    assert_combine_close("ll combined_x (capacity)", u16(out), refc)


def _random_shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        R = int(rng.choice([1, 2, 3, 5, 7, 8, 16, 24, 32]))
        E_loc = int(rng.integers(1, 9))
        E = R * E_loc
        K = int(rng.integers(1, min(8, E) + 1))
        routing = str(rng.choice(["uniform", "zipf", "replace"]))
        if routing != "replace" and K > E:
            K = E
        out.append(Workload(f"rand{i}", R=R, T=int(rng.integers(0, 300)), H=int(rng.choice([8, 16, 64, 264, 520])),
                            E=E, K=K, C=int(rng.integers(1, 41)), routing=routing,
                            mask=float(rng.choice([0.0, 0.2])), seed=int(rng.integers(0, 1000)),
                            expert_alignment=int(rng.choice([1, 2, 8]))))
    return out


@pytest.mark.parametrize("w", _random_shapes(24, 2024), ids=lambda w: f"{w.name}-R{w.R}T{w.T}K{w.K}E{w.E}H{w.H}C{w.C}")
def test_random_shapes_all_paths(w):
    """Seeded random shapes: bf16 path, low-latency layout and FP8 rows against the oracle."""
    full_parity(w, random_expert=True)
    cap = w.R * w.T * (w.K if w.routing == "replace" else 1)  # repeated experts need room per slot
    o = oracle.load()
    idx, wt, x = make_inputs(w)
    status, slot, rng_, cnt, rx, src, out = _ll_run(w, max(cap, 1), idx, wt, x.cuda())
    assert ep.ep_sync_status(status) == ep.EP_OK
    ref = oracle.ll_layout(o, w.R, w.T, w.K, w.E, max(cap, 1), idx.numpy())
    assert_equal("ll slot_pos", slot.cpu().numpy(), ref["slot_pos"])
    assert_equal("ll layout_range", rng_.cpu().numpy(), ref["layout_range"])
    refc = oracle.ll_combine(o, w.R, w.T, w.K, w.E, w.H, max(cap, 1), u16(rx), idx.numpy(), wt.numpy(),
                             ref["slot_pos"])
    assert_combine_close("ll combined_x", u16(out), refc)
    if w.H % 16 == 0:
        sh, lay, nt, status = run_layout_notify(w, idx)
        g = torch.Generator().manual_seed(w.seed)
        xb = torch.randint(0, 256, (w.R, w.T, w.H), generator=g, dtype=torch.uint8)
        xs = torch.randn(w.R, w.T, 3, generator=g)
        capr = max(1, worst_case_rows(w))
        r8 = torch.empty(capr, w.H, dtype=torch.uint8, device="cuda")
        rs = torch.empty(capr, 3, dtype=torch.float32, device="cuda")
        ep.ep_dispatch_fp8(sh, xb.cuda(), xs.cuda(), None, None, nt["send_pos"], nt["recv_base"], r8, rs,
                           None, None, None, status)
        assert ep.ep_sync_status(status) == ep.EP_OK
        lay_ref = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
        nt_ref = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay_ref)
        d8 = o.dispatch_fp8(w.R, w.T, w.K, w.E, w.H, w.C, xb.numpy(), xs.numpy(), idx.numpy(), wt.numpy(),
                            nt_ref["send_pos"], nt_ref["recv_base"], with_topk=False)
        rows = int(nt_ref["recv_base"][-1])
        assert_equal("fp8 recv_x", r8[:rows].cpu().numpy(), d8["recv_x"])
        assert_equal("fp8 recv_x_scales", rs[:rows].cpu().numpy(), d8["recv_x_scales"])
