"""ep_notify_dispatch_noalloc: the notify step for callers that cannot allocate
device memory (a host framework that owns every allocation, a serving loop
that forbids allocation after start-up), so they cannot pass a workspace.  It
uses a fixed scratch array inside the library instead.

Checked through the C ABI on consecutive calls, every output compared with the
CPU oracle and with the regular ep_notify_dispatch (which takes a caller
workspace).  The shapes are chosen so that every call takes notify's
decoupled-lookback path, the one that reads and writes the scratch (ticket
word and lookback words): the array keeps the previous call's contents, so a
call that failed to clear it would find words that look already published and
place rows wrongly on the second and third calls.  The middle call has another
shape, so the clear covers a range of another size.  This file is collected
last so a stop-at-first-failure run has already run everything else."""
import pytest
import torch

import oracle
from combine_get_dispatch_notify_gb300 import ep
from combine_get_dispatch_notify_gb300.workloads import CONFIGS, gen_routing

pytestmark = pytest.mark.gpu

# notify recounts sources directly (and leaves the scratch alone) when the
# membership rows of one source fit in 8 KB: T * R <= 8192
RECOUNT_LIMIT = 8 * 1024


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.lib()


def _shape(w):
    return ep.EpShape.make(w.R, w.T, w.K, w.E, w.H, w.C, w.expert_alignment)


def _layout(w, status, idx):
    sh = _shape(w)
    lay = ep.alloc_layout(sh)
    ep.ep_get_dispatch_layout(sh, idx.cuda(), lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
                              lay["num_tokens_per_expert"], lay["is_token_in_rank"], status)
    return sh, lay


def _outs(sh):
    return {k: torch.full(s, -7, dtype=dt, device="cuda") for k, (s, dt) in ep.notify_shapes(sh).items()}


def _compare_once(w, o):
    assert w.T * w.R > RECOUNT_LIMIT, f"{w.name} would not use the scratch"
    idx, _ = gen_routing(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sh, lay = _layout(w, status, idx)
    args = (lay["is_token_in_rank"], lay["num_tokens_per_rank"], lay["num_tokens_per_rdma_rank"],
            lay["num_tokens_per_expert"])
    got = _outs(sh)
    host = torch.full((w.R + 1,), -1, dtype=torch.int32).pin_memory()
    ep.ep_notify_dispatch_noalloc(sh, *args, got, status, host_num_recv_tokens=host)
    assert ep.ep_sync_status(status) == ep.EP_OK

    want = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, o.layout(w.R, w.T, w.K, w.E, idx.numpy()))
    for k in ep.notify_shapes(sh):
        g = got[k].cpu().numpy()
        assert (g == want[k]).all(), f"{w.name}: {k} differs from the oracle"

    ref = ep.alloc_notify(sh)
    ep.ep_notify_dispatch(sh, *args, ref, ref["workspace"], status)
    assert ep.ep_sync_status(status) == ep.EP_OK
    for k in ep.notify_shapes(sh):
        assert torch.equal(got[k], ref[k]), f"{w.name}: {k} differs from ep_notify_dispatch"
    want_host = torch.cat([ref["num_recv_tokens"], ref["recv_base"][-1:].to(torch.int32)]).cpu()
    assert torch.equal(host, want_host)


def test_noalloc_matches_oracle_on_consecutive_lookback_calls():
    o = oracle.load()
    # three calls in a row on the scratch: prefill, skewed (another shape), prefill again
    for name in ("prefill", "skewed", "prefill"):
        _compare_once(CONFIGS[name], o)


def test_noalloc_refuses_shapes_beyond_the_fixed_scratch():
    # 256 + R*C*(R+N)*8 bytes > 1 MiB for R=32, C=4096
    w = CONFIGS["large"].replace(T=4, C=4096)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, _ = gen_routing(w)
    sh, lay = _layout(w, status, idx)
    assert ep.ep_notify_workspace_bytes(sh) > (1 << 20)
    with pytest.raises(ep.EpError) as err:
        ep.ep_notify_dispatch_noalloc(sh, lay["is_token_in_rank"], lay["num_tokens_per_rank"],
                                      lay["num_tokens_per_rdma_rank"], lay["num_tokens_per_expert"],
                                      _outs(sh), status)
    assert err.value.status == ep.EP_ERR_INVALID_ARG
    assert ep.ep_sync_status(status) == ep.EP_OK  # nothing was enqueued
