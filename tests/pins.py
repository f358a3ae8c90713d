"""Pins for the CPU oracle: checks against facts the oracle does not compute itself.

Each ``check_*`` takes an oracle object and raises AssertionError when the
oracle disagrees with an independent fact:

* a hand-worked example (definitions applied by hand, derivation inline);
* a library routine the definition reduces to (numpy stable argsort / cumsum /
  bincount, torch's bf16 round-to-nearest-even);
* invariants and closed forms (counts add up, prefix rows end at the totals,
  combine of an identity expert equals bf16(n_dest * x), weights recombine);
* the exact result within the rounding error bound (fp64 reference sum).

The same checks run against deliberately broken oracle builds
(``ORACLE_MUTANT``) to show that each plausible mistake fails at least one.
"""
from __future__ import annotations

import numpy as np
import torch

from combine_get_dispatch_notify_gb300.workloads import Workload, gen_routing, gen_x
import oracle as oracle_mod
from oracle import bf16_bits_to_f32

NODE = 8


def nodes(R):
    return 1 if R <= NODE else R // NODE


def make_case(R, T, K, E, H, C, routing="uniform", mask=0.0, seed=0, align=1):
    w = Workload("case", R=R, T=T, H=H, E=E, K=K, C=C, routing=routing, mask=mask, seed=seed,
                 expert_alignment=align)
    idx, wt = gen_routing(w)
    x = gen_x(w).view(torch.int16).numpy().view(np.uint16)
    return w, idx.numpy(), wt.numpy(), x


def run(o, w, idx, wt, x, payload=True):
    lay = o.layout(w.R, w.T, w.K, w.E, idx)
    nt = o.notify(w.R, w.T, w.E, w.C, w.expert_alignment, lay)
    dp = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x, idx, wt, nt["send_pos"], nt["recv_base"],
                    payload=payload)
    return lay, nt, dp


def membership(R, E, idx):
    """is-token-in-rank built by scattering ones at each valid slot's owner rank."""
    Rr, T, K = idx.shape
    E_loc = E // R
    M = np.zeros((Rr, T, R), np.uint8)
    s_i, t_i, k_i = np.nonzero(idx >= 0)
    M[s_i, t_i, idx[s_i, t_i, k_i] // E_loc] = 1
    return M


# a few shapes that cover several nodes, ragged channels, masks and repeats
SHAPES = [
    dict(R=1, T=9, K=3, E=5, H=8, C=2, routing="replace", mask=0.2),
    dict(R=2, T=13, K=2, E=8, H=16, C=3),
    dict(R=4, T=17, K=3, E=8, H=8, C=5, routing="replace", mask=0.3),
    dict(R=8, T=21, K=4, E=32, H=8, C=4, mask=0.1),
    dict(R=16, T=11, K=8, E=64, H=8, C=3, routing="zipf", mask=0.1),
    dict(R=32, T=7, K=8, E=256, H=8, C=2, mask=0.1),
    dict(R=16, T=6, K=4, E=32, H=8, C=9, routing="replace"),  # C > T: empty channels
]


# --------------------------------------------------------------------------- hand-worked
def check_hand_worked(o):
    """R=2, T=4, K=2, E=4 (2 experts per rank), C=2 (channels [0,2) and [2,4)), H=2.

    Routing (expert ids per token, -1 = empty slot):
      rank 0: t0 [0,3] -> ranks {0,1}; t1 [1,-1] -> {0}; t2 [2,3] -> {1}; t3 [-1,-1] -> {}
      rank 1: t0 [3,2] -> {1};   t1 [0,2] -> {0,1}; t2 [1,0] -> {0}; t3 [2,-1] -> {1}
    """
    idx = np.array([[[0, 3], [1, -1], [2, 3], [-1, -1]],
                    [[3, 2], [0, 2], [1, 0], [2, -1]]], np.int64)
    wt = np.array([[[.5, .25], [1., 2.], [3., 4.], [5., 6.]],
                   [[7., 8.], [9., 10.], [11., 12.], [13., 14.]]], np.float32)
    x = np.arange(2 * 4 * 2, dtype=np.float32).reshape(2, 4, 2) + 1.0  # small integers: exact in bf16
    xb = o.f32_to_bf16(x)
    lay = o.layout(2, 4, 2, 4, idx)
    # expert 0 is hit by rank 0's t0 once, by rank 1's t1 and t2 (twice), ...
    np.testing.assert_array_equal(lay["num_tokens_per_expert"], [[1, 1, 1, 2], [2, 1, 3, 1]])
    np.testing.assert_array_equal(lay["is_token_in_rank"],
                                  [[[1, 1], [1, 0], [0, 1], [0, 0]], [[0, 1], [1, 1], [1, 0], [0, 1]]])
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], [[2, 2], [2, 3]])
    np.testing.assert_array_equal(lay["num_tokens_per_rdma_rank"], [[3], [4]])  # one node
    nt = o.notify(2, 4, 4, 2, 1, lay)
    # channel 0 = tokens 0,1; channel 1 = tokens 2,3; inclusive over channels
    np.testing.assert_array_equal(nt["gbl_channel_prefix_matrix"],
                                  [[[2, 2], [1, 2]], [[1, 2], [2, 3]]])
    np.testing.assert_array_equal(nt["rdma_channel_prefix_matrix"], [[[2, 3]], [[2, 4]]])
    np.testing.assert_array_equal(nt["rank_prefix_matrix"], [[2, 2], [4, 5]])
    np.testing.assert_array_equal(nt["recv_gbl_rank_prefix_sum"], [[2, 4], [2, 5]])
    np.testing.assert_array_equal(nt["num_recv_tokens"], [4, 5])
    np.testing.assert_array_equal(nt["recv_rdma_rank_prefix_sum"], [[3], [4]])
    np.testing.assert_array_equal(nt["num_rdma_recv_tokens"], [3, 4])
    # rank 0 owns experts 0,1: 1+2 and 1+1; rank 1 owns 2,3: 1+3 and 2+1
    np.testing.assert_array_equal(nt["num_recv_tokens_per_expert"], [[3, 2], [4, 3]])
    np.testing.assert_array_equal(nt["recv_base"], [0, 4, 9])
    np.testing.assert_array_equal(nt["recv_channel_offset"], [[[0, 2], [2, 3]], [[0, 1], [2, 4]]])
    np.testing.assert_array_equal(nt["send_pos"],
                                  [[[0, 0], [1, -1], [-1, 1], [-1, -1]],
                                   [[-1, 2], [2, 3], [3, -1], [-1, 4]]])
    dp = o.dispatch(2, 4, 2, 4, 2, 2, xb, idx, wt, nt["send_pos"], nt["recv_base"])
    # rank 0 region: (0,0) (0,1) (1,1) (1,2); rank 1 region: (0,0) (0,2) (1,0) (1,1) (1,3)
    np.testing.assert_array_equal(dp["recv_src_info"],
                                  [[0, 0], [0, 1], [1, 1], [1, 2], [0, 0], [0, 2], [1, 0], [1, 1], [1, 3]])
    np.testing.assert_array_equal(dp["recv_topk_idx"],
                                  [[0, -1], [1, -1], [0, -1], [1, 0], [-1, 1], [0, 1], [1, 0], [-1, 0], [0, -1]])
    np.testing.assert_array_equal(dp["recv_topk_w"],
                                  [[.5, 0], [1, 0], [9, 0], [11, 12], [0, .25], [3, 4], [7, 8], [0, 10], [13, 0]])
    want_rows = x.reshape(8, 2)[[0, 1, 5, 6, 0, 2, 4, 5, 7]]
    np.testing.assert_array_equal(bf16_bits_to_f32(dp["recv_x"]), want_rows)
    cb = o.combine(2, 4, 2, 2, dp["recv_x"], dp["recv_topk_w"], nt["send_pos"], nt["recv_base"])
    n_dest = np.array([[2, 1, 1, 0], [1, 2, 1, 1]], np.float32)
    np.testing.assert_array_equal(bf16_bits_to_f32(cb["combined_x"]), x * n_dest[..., None])
    np.testing.assert_array_equal(cb["combined_w"], np.where(idx >= 0, wt, 0))


def check_channel_ranges_hand(o):
    """T=5, C=4: q = ceil(5/4) = 2 -> channels [0,2) [2,4) [4,5) [5,5) (the last is empty)."""
    idx = np.array([[[0], [0], [0], [0], [0]]], np.int64)  # R=1, every token to rank 0
    lay = o.layout(1, 5, 1, 1, idx)
    nt = o.notify(1, 5, 1, 4, 1, lay)
    np.testing.assert_array_equal(nt["gbl_channel_prefix_matrix"], [[[2, 4, 5, 5]]])
    np.testing.assert_array_equal(nt["recv_channel_offset"], [[[0, 2, 4, 5]]])
    # T=5, C=2: q = 3 -> [0,3) [3,5)
    nt = o.notify(1, 5, 1, 2, 1, lay)
    np.testing.assert_array_equal(nt["gbl_channel_prefix_matrix"], [[[3, 5]]])


# --------------------------------------------------------------------------- layout
def check_layout_library(o):
    """Counts equal numpy scatter / bincount formulations; invariants hold."""
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        lay = o.layout(w.R, w.T, w.K, w.E, idx)
        M = membership(w.R, w.E, idx)
        np.testing.assert_array_equal(lay["is_token_in_rank"], M)
        for s in range(w.R):
            ids = idx[s][idx[s] >= 0]
            np.testing.assert_array_equal(lay["num_tokens_per_expert"][s], np.bincount(ids, minlength=w.E))
        np.testing.assert_array_equal(lay["num_tokens_per_rank"], M.sum(1))
        N = nodes(w.R)
        per_node = M.reshape(w.R, w.T, N, w.R // N).any(-1).sum(1)
        np.testing.assert_array_equal(lay["num_tokens_per_rdma_rank"], per_node)
        # invariants: slots add up, rank counts add up to destinations
        assert (lay["num_tokens_per_expert"].sum(1) == (idx >= 0).sum((1, 2))).all()
        assert (lay["num_tokens_per_rank"].sum(1) == M.sum((1, 2))).all()
        assert (lay["num_tokens_per_rdma_rank"] <= lay["num_tokens_per_rank"].reshape(w.R, N, -1).sum(-1)).all()
        if w.R == 1:
            np.testing.assert_array_equal(lay["num_tokens_per_rank"][:, 0], (idx >= 0).any(-1).sum(1))


# --------------------------------------------------------------------------- notify
def check_notify_library(o):
    for sh in SHAPES:
        for align in (1, 3, 16):
            w, idx, wt, x = make_case(**sh, align=align)
            lay = o.layout(w.R, w.T, w.K, w.E, idx)
            nt = o.notify(w.R, w.T, w.E, w.C, align, lay)
            M = membership(w.R, w.E, idx)
            R, T, C, N = w.R, w.T, w.C, nodes(w.R)
            # row of (s,t) in r's region = tokens of r before it in (s,t) order: a cumsum
            flat = M.reshape(R * T, R).astype(np.int64)
            order = np.cumsum(flat, axis=0) - flat
            want = np.where(flat == 1, order, -1).reshape(R, T, R)
            np.testing.assert_array_equal(nt["send_pos"], want)
            np.testing.assert_array_equal(nt["rank_prefix_matrix"], np.cumsum(M.sum(1), axis=0))
            np.testing.assert_array_equal(nt["recv_gbl_rank_prefix_sum"], nt["rank_prefix_matrix"].T)
            np.testing.assert_array_equal(nt["num_recv_tokens"], M.sum((0, 1)))
            np.testing.assert_array_equal(nt["recv_base"], np.concatenate([[0], np.cumsum(M.sum((0, 1)))]))
            # last channel column = per-rank / per-node totals; rows never decrease
            np.testing.assert_array_equal(nt["gbl_channel_prefix_matrix"][:, :, -1], lay["num_tokens_per_rank"])
            np.testing.assert_array_equal(nt["rdma_channel_prefix_matrix"][:, :, -1],
                                          lay["num_tokens_per_rdma_rank"])
            assert (np.diff(nt["gbl_channel_prefix_matrix"], axis=-1) >= 0).all()
            # block offsets: first row of channel c of s = tokens before the channel's first token
            q = -(-T // C) if T else 1
            for c in range(C):
                t0 = min(c * q, T)
                before = (np.cumsum(np.concatenate([np.zeros((1, R), np.int64), flat]), axis=0)
                          .reshape(-1, R))
                for s in range(R):
                    np.testing.assert_array_equal(nt["recv_channel_offset"][:, s, c], before[s * T + t0])
            # node-level receive prefix: tokens from the same-GPU-index peer of each node
            Mn = M.reshape(R, T, N, R // N).any(-1)  # [src, t, node]
            for r in range(R):
                run = 0
                for m in range(N):
                    peer = m * NODE + r % NODE
                    run += int(Mn[peer, :, r // NODE].sum())
                    assert nt["recv_rdma_rank_prefix_sum"][r, m] == run
            if R > NODE:  # the eight lanes of a node together receive every token entering it
                for n in range(N):
                    assert nt["num_rdma_recv_tokens"][n * NODE:(n + 1) * NODE].sum() == Mn[:, :, n].sum()
            # per-expert: sums over sources, rounded up to the alignment
            raw = np.zeros(w.E, np.int64)
            for s in range(R):
                raw += np.bincount(idx[s][idx[s] >= 0], minlength=w.E)
            got = nt["num_recv_tokens_per_expert"].reshape(-1).astype(np.int64)
            assert (got % align == 0).all()
            assert ((got - raw >= 0) & (got - raw < align)).all()


def check_channel_independence(o):
    """With contiguous channels the receive order does not depend on C."""
    w, idx, wt, x = make_case(R=8, T=23, K=3, E=16, H=8, C=1, mask=0.2)
    lay = o.layout(w.R, w.T, w.K, w.E, idx)
    ref = o.notify(w.R, w.T, w.E, 1, 1, lay)["send_pos"]
    for C in (2, 3, 5, 7, 23, 30):
        np.testing.assert_array_equal(o.notify(w.R, w.T, w.E, C, 1, lay)["send_pos"], ref)
    # equal-sized channels: per-channel counts from a plain reshape
    for C in (1, 23):
        nt = o.notify(w.R, w.T, w.E, C, 1, lay)
        M = lay["is_token_in_rank"].astype(np.int64)
        per = M.reshape(w.R, C, w.T // C, w.R).sum(2)  # [s, c, r]
        np.testing.assert_array_equal(nt["gbl_channel_prefix_matrix"], np.cumsum(per, axis=1).transpose(0, 2, 1))


# --------------------------------------------------------------------------- dispatch
def check_dispatch_stable_sort(o):
    """The pool is the stable sort by destination of (s, t, r) triples in (s, t) order."""
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        lay, nt, dp = run(o, w, idx, wt, x)
        M = membership(w.R, w.E, idx)
        s_i, t_i, r_i = np.nonzero(M)  # row-major: (s, t, r) order
        perm = np.argsort(r_i, kind="stable")
        want = np.stack([s_i[perm], t_i[perm]], 1)
        np.testing.assert_array_equal(dp["recv_src_info"], want)
        np.testing.assert_array_equal(dp["recv_x"], x[s_i[perm], t_i[perm]])
        assert int(nt["recv_base"][-1]) == len(perm) == int(lay["num_tokens_per_rank"].sum())


def check_dispatch_counting_sort(o):
    """K = 1: dispatch is a counting sort of tokens by owner rank."""
    w, idx, wt, x = make_case(R=8, T=40, K=1, E=16, H=8, C=3, mask=0.25)
    lay, nt, dp = run(o, w, idx, wt, x)
    flat = idx.reshape(-1)
    keep = np.nonzero(flat >= 0)[0]
    owner = flat[keep] // w.E_loc
    order = keep[np.argsort(owner, kind="stable")]
    np.testing.assert_array_equal(dp["recv_src_info"], np.stack([order // w.T, order % w.T], 1))
    # each received row carries exactly one local id: the token's expert minus the rank's first
    np.testing.assert_array_equal(dp["recv_topk_idx"][:, 0], flat[order] - np.sort(owner) * w.E_loc)


def check_dispatch_identity_rank(o):
    """R = 1: the pool is x restricted to tokens with a valid slot, in order."""
    w, idx, wt, x = make_case(R=1, T=30, K=2, E=4, H=16, C=4, mask=0.4)
    lay, nt, dp = run(o, w, idx, wt, x)
    keep = (idx[0] >= 0).any(-1)
    np.testing.assert_array_equal(dp["recv_x"], x[0][keep])
    np.testing.assert_array_equal(dp["recv_topk_idx"], idx[0][keep])


def check_dispatch_topk_fields(o):
    """Every valid slot lands once, as a local id on its owner; weights recombine exactly."""
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        lay, nt, dp = run(o, w, idx, wt, x)
        R, T, K = w.R, w.T, w.K
        assert ((dp["recv_topk_idx"] == -1) | ((dp["recv_topk_idx"] >= 0) & (dp["recv_topk_idx"] < w.E_loc))).all()
        rank_of_row = np.searchsorted(nt["recv_base"], np.arange(int(nt["recv_base"][-1])), side="right") - 1
        glob = np.where(dp["recv_topk_idx"] >= 0, dp["recv_topk_idx"] + rank_of_row[:, None] * w.E_loc, -1)
        wsum = np.zeros((R, T, K), np.float32)
        seen = np.zeros((R, T, K), np.int64)
        for p, (s, t) in enumerate(dp["recv_src_info"]):
            hit = glob[p] >= 0
            assert (glob[p][hit] == idx[s, t][hit]).all()
            seen[s, t] += hit
            wsum[s, t] += dp["recv_topk_w"][p]
        np.testing.assert_array_equal(seen, (idx >= 0).astype(np.int64))
        np.testing.assert_array_equal(wsum, np.where(idx >= 0, wt, 0))


# --------------------------------------------------------------------------- combine
def check_combine_identity_closed_form(o):
    """Identity expert: combine(dispatch(x)) = bf16(n_dest * x), n_dest <= 8 (exact fp32 sum)."""
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        lay, nt, dp = run(o, w, idx, wt, x)
        cb = o.combine(w.R, w.T, w.K, w.H, dp["recv_x"], dp["recv_topk_w"], nt["send_pos"], nt["recv_base"])
        n = membership(w.R, w.E, idx).sum(-1).astype(np.float32)
        xf = torch.from_numpy(bf16_bits_to_f32(x))
        want = (xf * torch.from_numpy(n)[..., None]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        want = np.where(n[..., None] == 0, np.uint16(0), want)  # no destination: +0, not x * 0
        np.testing.assert_array_equal(cb["combined_x"], want)
        np.testing.assert_array_equal(cb["combined_w"], np.where(idx >= 0, wt, 0))


def check_combine_error_bound(o):
    """Random expert outputs: within fp32-sum + one bf16 rounding of the fp64 sum."""
    rng = np.random.default_rng(7)
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        lay, nt, dp = run(o, w, idx, wt, x)
        rows = int(nt["recv_base"][-1])
        y = o.f32_to_bf16(rng.standard_normal((rows, w.H)).astype(np.float32) * 4)
        yw = rng.standard_normal((rows, w.K)).astype(np.float32)
        cb = o.combine(w.R, w.T, w.K, w.H, y, yw, nt["send_pos"], nt["recv_base"])
        yf = bf16_bits_to_f32(y).astype(np.float64)
        got = bf16_bits_to_f32(cb["combined_x"]).astype(np.float64)
        for s in range(w.R):
            for t in range(w.T):
                pos = nt["send_pos"][s, t]
                rr = [int(nt["recv_base"][r] + pos[r]) for r in range(w.R) if pos[r] >= 0]
                exact = yf[rr].sum(0) if rr else np.zeros(w.H)
                mag = np.abs(yf[rr]).sum(0) if rr else np.zeros(w.H)
                bound = 2.0 ** -8 * np.abs(exact) + (len(rr) * 2.0 ** -23) * mag + 1e-30
                assert (np.abs(got[s, t] - exact) <= bound).all(), (s, t)
                assert (np.abs(got[s, t] - exact) <= 1e-2 + 8e-3 * np.abs(exact)).all()
                wexact = yw.astype(np.float64)[rr].sum(0) if rr else np.zeros(w.K)
                wmag = np.abs(yw.astype(np.float64)[rr]).sum(0) if rr else np.zeros(w.K)
                assert (np.abs(cb["combined_w"][s, t] - wexact) <= len(rr) * 2.0 ** -23 * wmag + 1e-30).all()


def check_combine_order(o):
    """Ascending rank order decides the fp32 result: (2^24 + 1) - 2^24 = 0, not 1.

    Token (0,0) reaches ranks 0, 1, 2 with rows 2^24, 1, -2^24.  In ascending
    order 0 + 2^24 = 2^24; 2^24 + 1 is a tie between 2^24 and 2^24 + 2 and
    rounds to the even 2^24; adding -2^24 gives 0.  Descending order gives
    -2^24 + 1 = -16777215 (exact), then + 2^24 = 1.
    """
    idx = np.array([[[0, 1, 2]], [[-1, -1, -1]], [[-1, -1, -1]]], np.int64)  # R=3, T=1, K=3, E=3
    lay = o.layout(3, 1, 3, 3, idx)
    nt = o.notify(3, 1, 3, 1, 1, lay)
    y = o.f32_to_bf16(np.array([[2.0 ** 24], [1.0], [-(2.0 ** 24)]], np.float32))
    cb = o.combine(3, 1, 3, 1, y, None, nt["send_pos"], nt["recv_base"])
    assert bf16_bits_to_f32(cb["combined_x"])[0, 0, 0] == 0.0
    assert cb["combined_x"][1, 0, 0] == 0 and cb["combined_x"][2, 0, 0] == 0  # no destination -> +0


def check_combine_weight_order(o):
    """The combined weights are summed in ascending rank order as well.

    Token (0,0) reaches ranks 0, 1, 2 and the expert returns weight rows
    2^24, 1, -2^24 for slot 0.  Ascending: 2^24 + 1 ties to the even 2^24,
    minus 2^24 gives 0.  Descending: -2^24 + 1 = -16777215 (exact), plus 2^24
    gives 1.  Slot 1 gets 1, 2^-24, -1: ascending (1 + 2^-24) rounds to 1 (a
    tie to even), then 0; descending gives 2^-24 exactly, so any order but
    the ascending one shows in at least one slot.
    """
    idx = np.array([[[0, 1, 2]], [[-1, -1, -1]], [[-1, -1, -1]]], np.int64)  # R=3, T=1, K=3, E=3
    lay = o.layout(3, 1, 3, 3, idx)
    nt = o.notify(3, 1, 3, 1, 1, lay)
    y = o.f32_to_bf16(np.zeros((3, 1), np.float32))
    yw = np.array([[2.0 ** 24, 1.0, 0.0], [1.0, 2.0 ** -24, 0.0], [-(2.0 ** 24), -1.0, 0.0]], np.float32)
    cb = o.combine(3, 1, 3, 1, y, yw, nt["send_pos"], nt["recv_base"])
    np.testing.assert_array_equal(cb["combined_w"][0, 0], np.array([0.0, 0.0, 0.0], np.float32))
    assert (cb["combined_w"][1:] == 0).all()  # no destination: weights combine to +0


def check_bf16_rounding(o):
    """The oracle's fp32 -> bf16 rounding equals torch's round-to-nearest-even."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    # add exact ties, both parities, and the special values
    ties = (np.arange(0, 4096, dtype=np.uint32) << 16) | 0x8000
    specials = np.array([0, 0x80000000, 0x7f800000, 0xff800000, 0x7f7fffff, 0x7f7f8000, 0x00000001,
                         0x007fffff, 0x3f808000, 0x3f818000], np.uint32)
    bits = np.concatenate([bits, ties, ties | 0x80000000, specials])
    f = bits.view(np.float32)
    got = o.f32_to_bf16(f)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert np.isnan(bf16_bits_to_f32(got[nan])).all()


def check_dispatch_cached_mode(o):
    """Cached mode moves the same rows and source info, without top-k fields."""
    for sh in SHAPES[:4]:
        w, idx, wt, x = make_case(**sh)
        lay, nt, dp = run(o, w, idx, wt, x)
        cached = o.dispatch(w.R, w.T, w.K, w.E, w.H, w.C, x, idx, wt, nt["send_pos"], nt["recv_base"],
                            with_topk=False)
        assert cached["recv_topk_idx"] is None and cached["recv_topk_w"] is None
        np.testing.assert_array_equal(cached["recv_x"], dp["recv_x"])
        np.testing.assert_array_equal(cached["recv_src_info"], dp["recv_src_info"])


def check_dispatch_fp8(o):
    """FP8 rows and their scales land where the stable sort puts the token."""
    rng = np.random.default_rng(11)
    for sh in SHAPES:
        w, idx, wt, x = make_case(**{**sh, "H": 16})
        xb = rng.integers(0, 256, size=(w.R, w.T, w.H), dtype=np.uint8)
        xs = rng.standard_normal((w.R, w.T, 3)).astype(np.float32)
        lay, nt, dp = run(o, w, idx, wt, x)
        f8 = o.dispatch_fp8(w.R, w.T, w.K, w.E, w.H, w.C, xb, xs, idx, wt, nt["send_pos"], nt["recv_base"])
        M = membership(w.R, w.E, idx)
        s_i, t_i, r_i = np.nonzero(M)
        perm = np.argsort(r_i, kind="stable")
        np.testing.assert_array_equal(f8["recv_x"], xb[s_i[perm], t_i[perm]])
        np.testing.assert_array_equal(f8["recv_x_scales"], xs[s_i[perm], t_i[perm]])
        np.testing.assert_array_equal(f8["recv_topk_idx"], dp["recv_topk_idx"])
        np.testing.assert_array_equal(f8["recv_src_info"], dp["recv_src_info"])


# --------------------------------------------------------------------------- LL packed layout
def check_ll_layout_library(o):
    """Row of each slot in its expert's buffer = its rank in a stable sort by expert
    of the (source, token, slot) sequence; ranges and counts from bincount/cumsum."""
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        R, T, K, E = w.R, w.T, w.K, w.E
        cap = R * T * K
        ll = oracle_mod.ll_layout(o, R, T, K, E, cap, idx)
        flat = idx.reshape(-1)
        valid = np.nonzero(flat >= 0)[0]
        order = valid[np.argsort(flat[valid], kind="stable")]
        want = np.full(flat.shape, -1, np.int64)
        keys = flat[order]
        starts = np.searchsorted(keys, keys, side="left")
        want[order] = np.arange(len(order)) - starts
        np.testing.assert_array_equal(ll["slot_pos"].reshape(-1), want)
        per = np.stack([np.bincount(idx[s_][idx[s_] >= 0], minlength=E) for s_ in range(R)])  # [s, e]
        np.testing.assert_array_equal(ll["count"], per.sum(0))
        begin = np.cumsum(per, axis=0) - per
        np.testing.assert_array_equal(ll["layout_range"][:, :, 0], begin.T)
        np.testing.assert_array_equal(ll["layout_range"][:, :, 1], per.T)
        assert not ll["dropped"]


def check_ll_dispatch_and_combine(o):
    """LL dispatch places x rows where the layout says; combine with unit weights
    is bf16(n * x) (exact fp32 sum); random weights stay within the fp64 bound."""
    rng = np.random.default_rng(13)
    for sh in SHAPES:
        w, idx, wt, x = make_case(**sh)
        R, T, K, E, H = w.R, w.T, w.K, w.E, w.H
        cap = R * T * K
        ll = oracle_mod.ll_layout(o, R, T, K, E, cap, idx)
        dp = oracle_mod.ll_dispatch(o, R, T, K, E, H, cap, x, idx, ll["slot_pos"])
        ss, tt, kk = np.nonzero(idx >= 0)
        ee, rr = idx[ss, tt, kk], ll["slot_pos"][ss, tt, kk]
        np.testing.assert_array_equal(dp["recv_x"][ee, rr], x[ss, tt])
        np.testing.assert_array_equal(dp["recv_src_info"][ee, rr], np.stack([ss, tt], 1))
        assert (dp["recv_src_info"][..., 0] >= 0).sum() == len(ss)  # every slot lands once
        ones = np.ones_like(wt)
        cx = oracle_mod.ll_combine(o, R, T, K, E, H, cap, dp["recv_x"], idx, ones, ll["slot_pos"])
        n = (idx >= 0).sum(-1).astype(np.float32)
        xf = torch.from_numpy(bf16_bits_to_f32(x))
        want = (xf * torch.from_numpy(n)[..., None]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        want = np.where(n[..., None] == 0, np.uint16(0), want)
        np.testing.assert_array_equal(cx, want)
        y = o.f32_to_bf16(rng.standard_normal((E, cap, H)).astype(np.float32))
        wr = rng.standard_normal((R, T, K)).astype(np.float32)
        cx = oracle_mod.ll_combine(o, R, T, K, E, H, cap, y, idx, wr, ll["slot_pos"])
        yf = bf16_bits_to_f32(y).astype(np.float64)
        got = bf16_bits_to_f32(cx).astype(np.float64)
        terms = np.zeros((R, T, K, H))
        for s_, t_, k_ in zip(ss, tt, kk):
            terms[s_, t_, k_] = float(wr[s_, t_, k_]) * yf[idx[s_, t_, k_], ll["slot_pos"][s_, t_, k_]]
        exact = terms.sum(2)
        bound = 2.0 ** -8 * np.abs(exact) + K * 2.0 ** -23 * np.abs(terms).sum(2) + 1e-30
        assert (np.abs(got - exact) <= bound).all()


def check_ll_combine_order_and_fma(o):
    """Hand cases, R=1, T=1, E=3 experts, one slot each (cap 1).

    Order: y = 2^24, 1, -2^24 with unit weights in slots 0,1,2 -> (2^24+1)-2^24
    rounds to 0 in ascending slot order (1 in descending).
    Fused multiply-add: slot 0 w=-1, y=1+2^-7; slot 1 w=1+2^-23, y=1+2^-7.
    The exact product of slot 1 is 1+2^-7+2^-23+2^-30; with one rounding per
    fused step the sum is 2^-23+2^-30 = 2^-23(1+2^-7) (a bf16 value); a
    separate multiply would drop 2^-30 first and give 2^-23.
    """
    idx = np.array([[[0, 1, 2]]], np.int64)
    ll = oracle_mod.ll_layout(o, 1, 1, 3, 3, 1, idx)
    y = o.f32_to_bf16(np.array([[[2.0 ** 24]], [[1.0]], [[-(2.0 ** 24)]]], np.float32))
    cx = oracle_mod.ll_combine(o, 1, 1, 3, 3, 1, 1, y, idx, np.ones((1, 1, 3), np.float32), ll["slot_pos"])
    assert bf16_bits_to_f32(cx)[0, 0, 0] == 0.0
    y = o.f32_to_bf16(np.array([[[1 + 2.0 ** -7]], [[1 + 2.0 ** -7]], [[0.0]]], np.float32))
    wts = np.array([[[-1.0, 1 + 2.0 ** -23, 0.0]]], np.float32)
    cx = oracle_mod.ll_combine(o, 1, 1, 3, 3, 1, 1, y, idx, wts, ll["slot_pos"])
    assert bf16_bits_to_f32(cx)[0, 0, 0] == np.float32(2.0 ** -23 * (1 + 2.0 ** -7))


def check_ll_capacity_drop(o):
    """Slots whose row would reach the buffer size are dropped (-1), the rest keep their rows."""
    w, idx, wt, x = make_case(R=4, T=20, K=3, E=8, H=8, C=2)
    full = oracle_mod.ll_layout(o, 4, 20, 3, 8, 4 * 20 * 3, idx)
    small = oracle_mod.ll_layout(o, 4, 20, 3, 8, 5, idx)
    keep = full["slot_pos"] < 5
    np.testing.assert_array_equal(small["slot_pos"][keep], full["slot_pos"][keep])
    assert (small["slot_pos"][~keep] == -1).all() and small["dropped"] == (~keep & (idx >= 0)).any()


ALL_CHECKS = [
    check_hand_worked, check_channel_ranges_hand, check_layout_library, check_notify_library,
    check_channel_independence, check_dispatch_stable_sort, check_dispatch_counting_sort,
    check_dispatch_identity_rank, check_dispatch_topk_fields, check_combine_identity_closed_form,
    check_combine_error_bound, check_combine_order, check_combine_weight_order, check_bf16_rounding, check_dispatch_cached_mode,
    check_dispatch_fp8, check_ll_layout_library, check_ll_dispatch_and_combine,
    check_ll_combine_order_and_fma, check_ll_capacity_drop,
]
