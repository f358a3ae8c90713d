"""ep_layout_notify (layout and notify in one call) vs the CPU oracle, element
by element, through the C ABI: the cluster form on the shapes it takes (R <= 16,
T <= 1024, R*T <= 8192), the tiled form on the others, and the tiled form forced on every
case with several tile sizes (ep_debug_layout_notify_tiled); all bit-exact."""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import CONFIGS, Workload, gen_routing
from gpu_util import check_layout_notify, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.lib()


def _fused_expected(w: Workload) -> int:
    return 1 if (w.R <= 16 and w.T <= 1024 and w.R * w.T <= 8192) else 2


def _run(w: Workload, idx: torch.Tensor, host=None):
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    # poison the outputs: every element must be written by the call
    for d in (lay, nt):
        for k, v in d.items():
            if k != "workspace":
                v.fill_(0x5A if v.dtype == torch.uint8 else -7)
    ws = ep.alloc_layout_notify_workspace(sh)
    ep.ep_layout_notify(sh, idx.cuda(), lay, nt, ws, status, host)
    nt["workspace"] = ws
    return sh, lay, nt, status


def _oracle(w: Workload, idx: torch.Tensor):
    o = oracle.load()
    lay = o.layout(w.R, w.T, w.K, w.E, idx.numpy())
    nt = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay)
    return lay, nt


CASES = {
    "tiny": CONFIGS["tiny"],
    "low_latency": CONFIGS["low_latency"],
    "prefill": CONFIGS["prefill"],
    "skewed": CONFIGS["skewed"],
    "large": CONFIGS["large"],
    "single_rank": Workload("e", R=1, T=37, H=64, E=6, K=3, C=4, routing="replace", mask=0.2),
    "empty_tokens": Workload("e", R=4, T=0, H=64, E=8, K=2, C=3),
    "channels_exceed_tokens": Workload("e", R=8, T=50, H=128, E=64, K=4, C=64, mask=0.1),
    "odd_ranks_align": Workload("e", R=3, T=41, H=72, E=9, K=2, C=5, expert_alignment=4),
    "ragged_tokens_r16": Workload("e", R=16, T=1001, H=64, E=256, K=7, C=13, routing="zipf", mask=0.05),
    "max_experts": Workload("e", R=16, T=300, H=64, E=8192, K=9, C=4, routing="replace"),
    "r5_odd_topk": Workload("e", R=5, T=257, H=64, E=40, K=5, C=9, mask=0.3),
    "t8193": Workload("e", R=2, T=8193, H=64, E=16, K=2, C=3),
    "r32_small": Workload("e", R=32, T=19, H=8, E=256, K=8, C=3, routing="replace", mask=0.3),
    "all_masked": Workload("e", R=8, T=40, H=64, E=16, K=4, C=4, mask=1.0),
    "k32_repeats": Workload("e", R=16, T=97, H=64, E=512, K=32, C=7, routing="replace", mask=0.1),
    "c4096": Workload("e", R=4, T=300, H=64, E=16, K=2, C=4096, mask=0.2),
    "one_token": Workload("e", R=16, T=1, H=64, E=16, K=3, C=1),
    "one_expert_per_rank": Workload("e", R=16, T=200, H=64, E=16, K=5, C=3, routing="replace"),
    "r8_t8192_e2048": Workload("e", R=8, T=8192, H=64, E=2048, K=8, C=24, routing="zipf"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layout_notify_matches_oracle(name):
    w = CASES[name]
    idx, _ = gen_routing(w)
    lay_ref, nt_ref = _oracle(w, idx)
    sh, lay, nt, status = _run(w, idx)
    assert ep.ep_layout_notify_fused(sh) == _fused_expected(w)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    # a second call on the same buffers gives byte-identical results
    snap = {k: v.clone() for k, v in {**lay, **nt}.items() if k != "workspace"}
    ep.ep_layout_notify(sh, idx.cuda(), lay, nt, nt["workspace"], status)
    assert ep.ep_sync_status(status) == ep.EP_OK
    for k, v in snap.items():
        assert torch.equal(v, {**lay, **nt}[k]), f"{k} differs between calls"


def test_layout_notify_host_mapped_counts():
    w = CONFIGS["low_latency"]
    idx, _ = gen_routing(w)
    _, nt_ref = _oracle(w, idx)
    host = torch.zeros(w.R + 1, dtype=torch.int32).pin_memory()
    sh, lay, nt, status = _run(w, idx, host)
    torch.cuda.synchronize()
    assert ep.ep_sync_status(status) == ep.EP_OK
    want = np.concatenate([nt_ref["num_recv_tokens"], [nt_ref["recv_base"][-1]]]).astype(np.int32)
    assert np.array_equal(host.numpy(), want)


def test_layout_notify_bad_expert_id_reports_status():
    w = Workload("e", R=16, T=64, H=64, E=64, K=4, C=4)
    idx, _ = gen_routing(w)
    idx[3, 5, 1] = w.E + 7
    idx[9, 0, 0] = -5
    sh, lay, nt, status = _run(w, idx)
    assert ep.ep_sync_status(status) == ep.EP_ERR_INPUT
    # the bad ids are ignored: the counts are those of the top-k without them
    clean = idx.clone()
    clean[3, 5, 1] = -1
    clean[9, 0, 0] = -1
    lay_ref, nt_ref = _oracle(w, clean)
    check_layout_notify(lay, nt, lay_ref, nt_ref)


def test_layout_notify_feeds_dispatch():
    """The handle from the one-call form drives dispatch exactly like the
    handle from the two separate calls."""
    w = CONFIGS["low_latency"]
    idx, wt = gen_routing(w)
    o = oracle.load()
    sh, lay, nt, status = _run(w, idx)
    rows = int(nt["recv_base"][-1])
    x = torch.randn(w.R, w.T, w.H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    D = ep.alloc_dispatch(sh, rows)
    ep.ep_dispatch(sh, x.cuda(), idx.cuda(), wt.cuda(), nt["send_pos"], nt["recv_base"], D["recv_x"],
                   D["recv_topk_idx"], D["recv_topk_w"], D["recv_src_info"], status)
    assert ep.ep_sync_status(status) == ep.EP_OK
    lay_ref, nt_ref = _oracle(w, idx)
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x.view(torch.int16).numpy().view(np.uint16),
                    idx.numpy(), wt.numpy(), nt_ref["send_pos"], nt_ref["recv_base"])
    assert np.array_equal(D["recv_x"].view(torch.int16).cpu().numpy().view(np.uint16), dp["recv_x"])
    assert np.array_equal(D["recv_src_info"].cpu().numpy(), dp["recv_src_info"])


def test_layout_notify_first_call_inside_graph_capture():
    """A shape never seen before is first called inside a CUDA-graph capture
    (the one-kernel form's cluster-fit check runs then); replays match the oracle."""
    w = Workload("e", R=6, T=77, H=64, E=48, K=3, C=5, mask=0.1)
    idx, _ = gen_routing(w)
    lay_ref, nt_ref = _oracle(w, idx)
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay, nt = ep.alloc_layout(sh), ep.alloc_notify(sh)
    ws = ep.alloc_layout_notify_workspace(sh)
    idx_d = idx.cuda()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ep.ep_layout_notify(sh, idx_d, lay, nt, ws, status, stream=stream)
    for _ in range(2):
        for d in (lay, nt):
            for k, v in d.items():
                if k != "workspace":
                    v.fill_(-3 if v.dtype != torch.uint8 else 7)
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_sync_status(status) == ep.EP_OK
        check_layout_notify(lay, nt, lay_ref, nt_ref)
    assert ep.ep_layout_notify_fused(sh) == 1


@pytest.mark.parametrize("name", ["low_latency", "large_r32_small"])
def test_pipeline_replayed_from_a_cuda_graph(name):
    """The whole step captured once and replayed on new inputs copied into the
    same buffers: every output matches the oracle for each replay."""
    from combine_get_dispatch_notify_gb300.workloads import gen_x, worst_case_rows

    w = CONFIGS["low_latency"] if name == "low_latency" else Workload(
        "e", R=32, T=24, H=256, E=256, K=8, C=3, mask=0.1)  # tiled layout + notify
    o = oracle.load()
    sh = shape_of(w)
    pipe = ep.Pipeline(sh, max(1, worst_case_rows(w)))
    x_d = torch.empty(w.R, w.T, w.H, dtype=torch.bfloat16, device="cuda")
    idx_d = torch.empty(w.R, w.T, w.K, dtype=torch.int64, device="cuda")
    wt_d = torch.empty(w.R, w.T, w.K, dtype=torch.float32, device="cuda")
    idx0, wt0 = gen_routing(w)
    idx_d.copy_(idx0)
    wt_d.copy_(wt0)
    x_d.copy_(gen_x(w))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pipe.run(x_d, idx_d, wt_d, stream=stream)  # eager call first, as a server would at start-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cx, cw = pipe.run(x_d, idx_d, wt_d, stream=stream)
    for seed in (11, 12):
        ws = Workload(w.name, R=w.R, T=w.T, H=w.H, E=w.E, K=w.K, C=w.C, mask=w.mask, seed=seed)
        idx, wt = gen_routing(ws)
        x = gen_x(ws)
        idx_d.copy_(idx)
        wt_d.copy_(wt)
        x_d.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_sync_status(pipe.status) == ep.EP_OK
        xb = x.view(torch.int16).numpy().view(np.uint16)
        lay, nt, dp, cb = oracle.run_all(w.R, w.T, w.K, w.E, w.H, w.C, w.expert_alignment, xb, idx.numpy(),
                                         wt.numpy(), o)
        check_layout_notify(pipe.layout, pipe.notify, lay, nt)
        rows = int(nt["recv_base"][-1])
        assert np.array_equal(pipe.dispatch["recv_x"][:rows].view(torch.int16).cpu().numpy().view(np.uint16),
                              dp["recv_x"])
        assert np.array_equal(pipe.dispatch["recv_src_info"][:rows].cpu().numpy(), dp["recv_src_info"])
        assert np.array_equal(cx.view(torch.int16).cpu().numpy().view(np.uint16), cb["combined_x"])
        assert np.array_equal(cw.cpu().numpy(), cb["combined_w"])


# ----------------------------------------------------------------------------- tiled form
def _tiled(w: Workload, idx: torch.Tensor, tile_tokens=0, ws=None, stall=-1, limit_us=1000000):
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.alloc_layout(sh)
    nt = ep.alloc_notify(sh)
    for d in (lay, nt):
        for k, v in d.items():
            if k != "workspace":
                v.fill_(0x5A if v.dtype == torch.uint8 else -7)
    if ws is None:
        ws = ep.alloc_layout_notify_workspace(sh, nbytes=_tiled_ws_bytes(w, tile_tokens))
    ep.ep_debug_layout_notify_tiled(sh, idx.cuda(), lay, nt, ws, status, tile_tokens=tile_tokens,
                                    stall_tile=stall, wait_limit_us=limit_us)
    return sh, lay, nt, status, ws


def _tiled_ws_bytes(w: Workload, tile_tokens: int) -> int:
    """Workspace the tiled form needs with tiles of ``tile_tokens`` (0: default)."""
    sh = shape_of(w)
    if tile_tokens == 0:
        return ep.ep_layout_notify_workspace_bytes(sh)
    tiles = w.R * (max(1, -(-w.T // tile_tokens)) if w.T > 0 else 1)
    return 256 + (2 << 20) + (64 << 10) + (18 << 10) + 8 * (w.R + w.N) * tiles


TILED_SIZES = (32, 96, 512, 0)


@functools.lru_cache(maxsize=None)
def _case_ref(name: str):
    w = CASES[name]
    idx, _ = gen_routing(w)
    return idx, _oracle(w, idx)


@pytest.mark.parametrize("tile", TILED_SIZES, ids=lambda t: f"tile{t}")
@pytest.mark.parametrize("name", sorted(CASES))
def test_tiled_layout_notify_matches_oracle(name, tile):
    w = CASES[name]
    if tile == 32 and w.R * w.T > 200000:
        pytest.skip("32-token tiles of a full-size workload: covered by the larger tiles")
    idx, (lay_ref, nt_ref) = _case_ref(name)
    sh, lay, nt, status, ws = _tiled(w, idx, tile)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)


def test_tiled_workspace_serves_shapes_in_turn_and_stays_clean():
    """One workspace, sized for the largest, serves several shapes and tile
    sizes in turn; after every call its expert counters and per-source
    counters are zero again."""
    names = ["prefill", "r32_small", "ragged_tokens_r16", "empty_tokens", "prefill", "k32_repeats"]
    need = max(_tiled_ws_bytes(CASES[n], t) for n in names for t in (32, 0))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for i, n in enumerate(names):
        w = CASES[n]
        tile = 32 if i % 2 else 0
        idx, _ = gen_routing(w)
        lay_ref, nt_ref = _oracle(w, idx)
        sh, lay, nt, status, _ = _tiled(w, idx, tile, ws=ws)
        assert ep.ep_sync_status(status) == ep.EP_OK
        check_layout_notify(lay, nt, lay_ref, nt_ref)
        head = ws[:256].cpu()
        assert (head[8:16] == 0).all()                               # finished-tiles counter
        assert int((ws[256:256 + (2 << 20) + (64 << 10)] != 0).sum()) == 0  # expert counters
        seq = int(head[:8].numpy().view(np.uint64)[0]) >> 32                # this call's sequence number
        banks = 256 + (2 << 20) + (64 << 10)
        nxt = banks + ((seq + 1) & 1) * (9 << 10)
        assert int((ws[nxt:nxt + (9 << 10)] != 0).sum()) == 0               # the next call's source totals


def test_tiled_stall_times_out_and_next_call_is_exact():
    """A tile that never publishes its lookback words makes the tiles after it
    give up (EP_ERR_TIMEOUT, no hang); a normal call afterwards is bit-exact."""
    w = CASES["ragged_tokens_r16"]
    idx, _ = gen_routing(w)
    sh, lay, nt, status, ws = _tiled(w, idx, 64, stall=5, limit_us=2000)
    assert ep.ep_sync_status(status) == ep.EP_ERR_TIMEOUT
    lay_ref, nt_ref = _oracle(w, idx)
    status.zero_()
    ep.ep_debug_layout_notify_tiled(sh, idx.cuda(), lay, nt, ws, status, tile_tokens=64)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)


def test_tiled_first_call_inside_graph_capture():
    """The tiled form's first call for a shape inside a CUDA-graph capture (its
    occupancy query runs then); replays match the oracle."""
    w = Workload("e", R=24, T=413, H=64, E=96, K=6, C=7, mask=0.1)
    idx, _ = gen_routing(w)
    lay_ref, nt_ref = _oracle(w, idx)
    sh = shape_of(w)
    assert ep.ep_layout_notify_fused(sh) == 2
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay, nt = ep.alloc_layout(sh), ep.alloc_notify(sh)
    ws = ep.alloc_layout_notify_workspace(sh)
    idx_d = idx.cuda()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ep.ep_layout_notify(sh, idx_d, lay, nt, ws, status, stream=stream)
    for _ in range(3):
        for d in (lay, nt):
            for k, v in d.items():
                if k != "workspace":
                    v.fill_(-3 if v.dtype != torch.uint8 else 7)
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_sync_status(status) == ep.EP_OK
        check_layout_notify(lay, nt, lay_ref, nt_ref)


def test_tiled_refuses_bad_tile_sizes_and_small_workspace():
    w = CASES["r5_odd_topk"]
    idx, _ = gen_routing(w)
    sh = shape_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay, nt = ep.alloc_layout(sh), ep.alloc_notify(sh)
    ws = ep.alloc_layout_notify_workspace(sh)
    for bad in (16, 48 + 1, 8224):
        with pytest.raises(ep.EpError):
            ep.ep_debug_layout_notify_tiled(sh, idx.cuda(), lay, nt, ws, status, tile_tokens=bad)
    small = torch.zeros(ep.ep_layout_notify_workspace_bytes(sh) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ep.EpError):
        ep.ep_debug_layout_notify_tiled(sh, idx.cuda(), lay, nt, small, status)
    with pytest.raises(ValueError):
        ep.ep_layout_notify(sh, idx.cuda(), lay, nt, small, status)
    assert ep.ep_sync_status(status) == ep.EP_OK  # nothing was enqueued


def test_tiled_bad_expert_id_reports_status():
    """Ids outside [-1, E) in the tiled form: EP_ERR_INPUT, and every output is
    that of the top-k with those slots empty."""
    w = Workload("e", R=24, T=300, H=64, E=96, K=6, C=7, mask=0.1)
    idx, _ = gen_routing(w)
    idx[3, 5, 1] = w.E + 7
    idx[20, 299, 5] = -5
    sh, lay, nt, status, ws = _tiled(w, idx, 64)
    assert ep.ep_sync_status(status) == ep.EP_ERR_INPUT
    clean = idx.clone()
    clean[3, 5, 1] = -1
    clean[20, 299, 5] = -1
    lay_ref, nt_ref = _oracle(w, clean)
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    assert int((ws[256:256 + (2 << 20) + (64 << 10)] != 0).sum()) == 0


def test_tiled_every_expert_counter_in_use():
    """32 ranks and 8192 experts: the tiled form's expert counters are used in
    full ([32][8192]); results exact, counters left zero."""
    w = Workload("e", R=32, T=64, H=64, E=8192, K=16, C=3, routing="replace", mask=0.05)
    idx, _ = gen_routing(w)
    lay_ref, nt_ref = _oracle(w, idx)
    sh, lay, nt, status, ws = _tiled(w, idx, 32)
    assert ep.ep_sync_status(status) == ep.EP_OK
    check_layout_notify(lay, nt, lay_ref, nt_ref)
    assert int((ws[256:256 + (2 << 20) + (64 << 10)] != 0).sum()) == 0
