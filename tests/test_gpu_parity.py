"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small and ragged shapes are compared element by element on every output; the
four large workloads are compared element by element on sampled heads (each
head is an independent problem the oracle computes whole), with invariants
of the gradient checked on every head.
"""
import numpy as np
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
import workloads
from oracle import attention as A
from oracle import dag_sim as d

from _gpu import LSE_ABS_TOL, Problem, assert_close, err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


SMALL = [
    # B, H, S, D, causal, tile: several tiles, ragged tails, both head dims and tiles
    (1, 2, 256, 64, False, 64),
    (1, 2, 256, 64, True, 64),
    (1, 2, 512, 128, True, 128),
    (1, 1, 333, 64, True, 64),
    (1, 2, 700, 128, True, 128),
    (1, 2, 700, 128, False, 128),
    (2, 2, 640, 64, True, 128),
    (1, 3, 1000, 64, False, 128),
    (1, 1, 100, 128, True, 128),     # a single ragged tile
    (1, 1, 1, 64, False, 64),        # one query, one key
    (1, 2, 192, 128, False, 64),
]


def schedules_for(causal, S, tile):
    n = (S + tile - 1) // tile
    out = []
    for s in workloads.ALL_SCHEDULES:
        if s == "shift" and causal:
            continue
        if s == "symmetric_shift" and (not causal or n % 2):
            continue
        out.append(s)
    return out


@pytest.mark.parametrize("B,H,S,D,causal,tile", SMALL)
def test_forward_and_backward_match_oracle(B, H, S, D, causal, tile):
    P = Problem(B, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    dash.dash_sync_status()
    ro, rl = P.oracle_fwd()
    assert_close("O", o, ro)
    assert err(lse, rl)[1] <= LSE_ABS_TOL
    # end to end: oracle forward + backward from the bf16 inputs
    q, k, v, do = P.f64
    ref_e2e = A.backward(q, k, v, ro, do, rl, causal, P.scale)
    # isolated: oracle backward fed the GPU's O and LSE
    ref_iso = A.backward(q, k, v, o.double().cpu().numpy(), do, lse.double().cpu().numpy(), causal, P.scale)
    for sched in schedules_for(causal, S, tile):
        dq, dk, dv = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile)
        dash.dash_sync_status()
        for name, x, r1, r2 in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref_iso, ref_e2e):
            assert_close(f"{sched} {name} (isolated)", x, r1)
            assert_close(f"{sched} {name} (end to end)", x, r2)


@pytest.mark.parametrize("B,H,S,D,causal,tile", [SMALL[2], SMALL[5], SMALL[6], SMALL[7]])
def test_two_dq_chains_match_oracle(B, H, S, D, causal, tile):
    # the two-chain reduction (even and odd ranks in separate accumulators)
    # against the oracle, for every ordered schedule
    P = Problem(B, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    q, k, v, do = P.f64
    ref = A.backward(q, k, v, o.double().cpu().numpy(), do, lse.double().cpu().numpy(), causal, P.scale)
    for sched in schedules_for(causal, S, tile):
        if sched == "atomic":
            continue
        got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile, dq_chains=2)
        dash.dash_sync_status()
        for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(f"{sched} two chains {name}", x, r)


@pytest.mark.parametrize("S,causal,sched,H,ctas", [(256, False, "shift", 5, 10), (512, True, "symmetric_shift", 5, 10),
                                                   (300, False, "shift", 7, 12), (640, True, "symmetric_shift", 7, 12)])
def test_fill_small_matches_oracle(S, causal, sched, H, ctas):
    # fill (an extension) on a small CTA budget, so that some heads run on the
    # leftover CTAs: every head against the oracle, including a ragged tail
    tile, D = 64, 64
    n = (S + tile - 1) // tile
    _, _, used, hs, fill_sched, _ = dash.dash_build_shift_fill(H, n, causal, sched, ctas)
    assert hs < H and fill_sched is not None and used == ctas
    P = Problem(1, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    q, k, v, do = P.f64
    ref = A.backward(q, k, v, o.double().cpu().numpy(), do, lse.double().cpu().numpy(), causal, P.scale)
    got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile, num_ctas=ctas,
                        shift_fill=1)
    dash.dash_sync_status()
    for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_close(f"{sched} with fill {name}", x, r)
    again = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile, num_ctas=ctas,
                          shift_fill=1)
    dash.dash_sync_status()
    assert all(torch.equal(a, b) for a, b in zip(got, again))


@pytest.mark.parametrize("chains", [1, 2])
@pytest.mark.parametrize("wname,sched", [("full_s4096_d128", "shift"), ("causal_s8192_d64", "symmetric_shift")])
def test_fill_heads_equal_their_own_schedules(wname, sched, chains):
    # fill (an extension): the heads on whole gangs give the plain schedule's
    # bits, the heads on the leftover CTAs the fill schedule's; the last head
    # is also checked against the row-wise oracle on sampled rows
    w = workloads.WORKLOADS[wname]
    BH, n = w.B * w.H, w.S // w.tile
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, _, ctas, hs, fill_sched, _ = dash.dash_build_shift_fill(BH, n, w.causal, sched, sms)
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    run = lambda s_, **kw: [x.reshape(BH, w.S, w.D) for x in dash.attn_bwd(
        P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, s_, tile=w.tile, dq_accum=True, dq_chains=chains, **kw)]
    fill, plain = run(sched, shift_fill=1), run(sched)
    dash.dash_sync_status()
    for a, b in zip(fill, plain):
        assert torch.equal(a[:hs], b[:hs])
    if fill_sched:
        other = run(fill_sched)
        dash.dash_sync_status()
        for a, b in zip(fill, other):
            assert torch.equal(a[hs:], b[hs:])
    print(f"{wname} {sched} with fill on {sms} SMs: {hs} of {BH} heads, the rest {fill_sched}, {ctas} CTAs")
    q, k, v, do = P.f64
    b_, h_ = w.B - 1, w.H - 1
    rows = sorted({0, w.tile - 1, w.tile, w.S // 2 + 5, w.S - 1})
    oh, lh = o[b_, h_].double().cpu().numpy(), lse[b_, h_].double().cpu().numpy()
    ref = A.backward_rows(q[b_, h_], k[b_, h_], v[b_, h_], oh, do[b_, h_], lh, w.causal, P.scale, rows)
    for name, x, r in zip(("dQ", "dK", "dV"), fill[:3], ref):
        assert_close(f"{sched} with fill {name}[{b_},{h_}] rows", x[BH - 1][rows], r)


# split gangs (an extension): S, D, tile, mask, schedule, split; several
# sub-gangs per head, ragged tails, both head dims
SPLIT = [(512, 64, 64, False, "shift", 2), (500, 64, 64, False, "shift", 4),
         (1000, 64, 64, True, "symmetric_shift", 4), (1024, 128, 128, True, "symmetric_shift", 2),
         (700, 128, 128, False, "shift", 2)]


@pytest.mark.parametrize("S,D,tile,causal,sched,split", SPLIT,
                         ids=[f"{s}_s{S}_d{D}_k{k}" for S, D, _, _, s, k in SPLIT])
def test_split_gangs_match_oracle(S, D, tile, causal, sched, split):
    # every output against the oracle, with one and two dQ chains; the bits do
    # not depend on the CTA count (the library's choice, one sub-gang, three)
    H = 3
    n = (S + tile - 1) // tile
    g = (n // 2 if sched == "symmetric_shift" else n) // split
    P = Problem(1, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    q, k, v, do = P.f64
    ref = A.backward(q, k, v, o.double().cpu().numpy(), do, lse.double().cpu().numpy(), causal, P.scale)
    for chains in (1, 2):
        first = None
        for ctas in (0, g, 3 * g):
            got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile, dq_accum=True,
                                dq_chains=chains, shift_split=split, num_ctas=ctas)
            dash.dash_sync_status()
            if first is None:
                first = got
                for name, x, r in zip(("dQ", "dK", "dV"), got[:3], ref):
                    assert_close(f"{sched} split {split}, {chains} chain(s) {name}", x, r)
            else:
                assert all(torch.equal(a, b) for a, b in zip(first, got)), f"{ctas} CTAs changed the bits"


@pytest.mark.parametrize("wname,sched", [("full_s4096_d128", "shift"), ("causal_s8192_d64", "symmetric_shift")])
def test_split_gangs_full_size(wname, sched):
    # split gangs at full size as the library picks them (shift_split = -1):
    # the same bits as the chosen split asked for by name, and on a second
    # run; sampled rows of the first and last heads against the row-wise oracle
    w = workloads.WORKLOADS[wname]
    BH = w.B * w.H
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    k, ctas, _ = dash.dash_choose_split(BH, w.S // w.tile, w.causal, sched, sms)
    assert k >= 1
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    run = lambda kk, **kw: dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, tile=w.tile,
                                         shift_split=kk, **kw)
    got, again, named = run(-1), run(-1), run(k, num_ctas=ctas)
    dash.dash_sync_status()
    assert all(torch.equal(a, b) for a, b in zip(got, again))
    assert all(torch.equal(a, b) for a, b in zip(got, named))
    print(f"{wname} {sched}: split {k} on {ctas} CTAs")
    q, k, v, do = P.f64
    rows = sorted({0, w.tile - 1, w.tile, w.S // 2 + 5, w.S - 1})
    for b_, h_ in ((0, 0), (w.B - 1, w.H - 1)):
        oh, lh = o[b_, h_].double().cpu().numpy(), lse[b_, h_].double().cpu().numpy()
        ref = A.backward_rows(q[b_, h_], k[b_, h_], v[b_, h_], oh, do[b_, h_], lh, w.causal, P.scale, rows)
        for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(f"{sched} split {k} {name}[{b_},{h_}] rows", x[b_, h_][rows], r)


def test_split_gangs_run_shift_past_the_sm_count():
    # a shift gang of n = 256 chains is larger than the GPU: whole gangs cannot
    # run it (no CTA count holds one), split gangs can; sampled rows against
    # the row-wise oracle, and the same bits twice
    S, D = 32768, 64
    n = S // 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert n > sms and dash.dash_choose_ctas(1, n, False, "shift", sms) == -1
    P = Problem(1, 1, S, D, False)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, False, P.scale)
    with pytest.raises(dash.DashError):
        dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, "shift")
    k, ctas, _ = dash.dash_choose_split(1, n, False, "shift", sms)
    assert k > 1 and ctas % (n // k) == 0
    got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, "shift", shift_split=-1)
    again = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, "shift", shift_split=-1)
    dash.dash_sync_status()
    assert all(torch.equal(a, b) for a, b in zip(got, again))
    q, k_, v, do = P.f64
    rows = [0, 127, 128, S // 2 + 5, S - 1]
    ref = A.backward_rows(q[0, 0], k_[0, 0], v[0, 0], o[0, 0].double().cpu().numpy(), do[0, 0],
                          lse[0, 0].double().cpu().numpy(), False, P.scale, rows)
    for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_close(f"shift split {k} at n = {n} {name} rows", x[0, 0][rows], r)


TIMED = [(512, 64, 64, False, 5), (500, 64, 64, False, 7), (1000, 64, 64, True, 9), (1024, 128, 128, True, 5),
         (700, 128, 128, False, 4)]


@pytest.mark.parametrize("S,D,tile,causal,ctas", TIMED, ids=[f"s{S}_d{D}_{'causal' if c else 'full'}_p{p}"
                                                              for S, D, _, c, p in TIMED])
def test_timed_ranks_match_oracle(S, D, tile, causal, ctas):
    # timed ranks (an extension) for every ordered schedule of the mask, on the library's CTA count and on a
    # count that spreads the gangs over time, with one and two dQ chains; the same bits on a second run
    H = 3
    P = Problem(1, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    q, k, v, do = P.f64
    ref = A.backward(q, k, v, o.double().cpu().numpy(), do, lse.double().cpu().numpy(), causal, P.scale)
    n = (S + tile - 1) // tile
    for sched in schedules_for(causal, S, tile):
        if sched == "atomic":
            continue
        # timed ranks alone, and with split gangs of two where the gang divides
        gang = n // 2 if sched == "symmetric_shift" else n
        splits = (1, 2) if sched in ("shift", "symmetric_shift") and gang % 2 == 0 else (1,)
        for split in splits:
            for chains in (1, 2):
                for num in (0, ctas):
                    run = lambda: dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile,
                                                dq_chains=chains, rank_order=1, num_ctas=num, shift_split=split)
                    got, again = run(), run()
                    dash.dash_sync_status()
                    for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
                        assert_close(f"{sched} timed split {split}, {chains} chain(s), {num} CTAs {name}", x, r)
                    assert all(torch.equal(a, b) for a, b in zip(got, again))


@pytest.mark.parametrize("wname,sched", [("causal_s16384_d128", "symmetric_shift"), ("full_s4096_d128", "shift")])
def test_timed_ranks_full_size(wname, sched):
    # timed ranks on every SM at full size: sampled rows of the first and last heads against the row-wise oracle,
    # the same bits twice; dK and dV equal the pages' order's (they do not depend on the dQ order)
    w = workloads.WORKLOADS[wname]
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    run = lambda **kw: dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, tile=w.tile, **kw)
    got, again, plain = run(rank_order=1), run(rank_order=1), run()
    dash.dash_sync_status()
    assert all(torch.equal(a, b) for a, b in zip(got, again))
    assert torch.equal(got[1], plain[1]) and torch.equal(got[2], plain[2])
    q, k, v, do = P.f64
    rows = sorted({0, w.tile - 1, w.tile, w.S // 2 + 5, w.S - 1})
    for b_, h_ in ((0, 0), (w.B - 1, w.H - 1)):
        oh, lh = o[b_, h_].double().cpu().numpy(), lse[b_, h_].double().cpu().numpy()
        ref = A.backward_rows(q[b_, h_], k[b_, h_], v[b_, h_], oh, do[b_, h_], lh, w.causal, P.scale, rows)
        for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(f"{sched} timed {name}[{b_},{h_}] rows", x[b_, h_][rows], r)


def _red_add_f32(acc, x):
    """fp32 add as red.global.add.f32 performs it: round to nearest even, with
    subnormal inputs and results flushed to (signed) zero."""
    tiny = np.float32(np.finfo(np.float32).tiny)
    flush = lambda a: np.where(np.abs(a) < tiny, np.copysign(np.float32(0), a), a).astype(np.float32)
    return flush(flush(acc) + flush(x))


# (S, D, tile) of the order check: one case per kernel instantiation that the
# workloads use (D = 64 with 64- and 128-row tiles, D = 128 with 128-row tiles;
# the last two are the ones the large workloads run, with their stage counts
# and, at D = 128, dQ in the dP^T columns of tensor memory)
ORDER_CASES = [(256, 64, 64), (512, 128, 128), (512, 64, 128)]


@pytest.mark.parametrize("S,D,tile", ORDER_CASES, ids=[f"s{s}_d{d}_t{t}" for s, d, t in ORDER_CASES])
@pytest.mark.parametrize("causal", [False, True])
def test_kernel_adds_partials_in_table_rank_order(causal, S, D, tile):
    # The order check: each task's fp32 dQ partial is taken from a run whose
    # table holds that task alone (rank 0 stores its partial unchanged); the
    # CPU then adds the partials of every tile in the schedule's rank order in
    # fp32 (for two chains: even and odd ranks apart, then chain 0 + chain 1),
    # and the result must equal the accumulator of the whole run bit for bit.
    B, H = 1, 2
    n, BH = S // tile, B * H
    P = Problem(B, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    tiles = [(kv, q) for kv in range(n) for q in range(n) if not causal or q >= kv]
    part = {}
    for bh in range(BH):
        for kv, q in tiles:
            one = np.array([[bh, kv, q, dash.TASK_FIRST | dash.TASK_LAST]], dtype=np.int32)
            acc = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, "serial", tile=tile, dq_accum=True,
                                tasks=one, cta_off=np.array([0, 1], dtype=np.int32))[3]
            dash.dash_sync_status()
            part[(bh, kv, q)] = acc.reshape(BH, S, D)[bh, q * tile:(q + 1) * tile].cpu().numpy()
    cyclic = "symmetric_shift" if causal else "shift"
    # the pages' orders, split gangs of two (an extension) for the cyclic schedule, and timed ranks (an
    # extension) of the cyclic schedule on 3 CTAs, which spreads its gangs over time (ranks per head)
    for sched, split, timed in (("serial", 1, 0), ("descending_q", 1, 0), (cyclic, 1, 0), (cyclic, 2, 0),
                                (cyclic, 1, 1), (cyclic, 2, 1)):
        extra = {}
        if timed:
            tasks_t, _, _ = dash.dash_build_schedule_ex(BH, n, causal, sched, split, 1, 3)
            rank = {(int(b), int(kv), int(q)): int(w) & dash.TASK_RANK_MASK for b, kv, q, w in tasks_t}
            extra = {"rank_order": 1, "num_ctas": 3}
        else:
            if split == 1:
                chains_ = d.head_chains(sched, n, causal)
                ranked = zip(chains_, d.head_ranks(sched, n, causal, chains_))
            else:
                ranked = [(ch, rks) for _, ch, rks in d.split_chains(sched, 1, n, causal, split)]
            head_rank = {t: rk for ch, rks in ranked for t, rk in zip(ch, rks)}
            rank = {(bh, kv, q): head_rank[(kv, q)] for bh in range(BH) for kv, q in tiles}
        for nch in (1, 2):
            got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tile=tile, dq_accum=True,
                                dq_chains=nch, shift_split=split, **extra)[3]
            dash.dash_sync_status()
            got = got.reshape(BH, S, D).cpu().numpy()
            for bh in range(BH):
                for q in range(n):
                    order = sorted((rank[(bh, kv, q)], kv) for kv, qq in tiles if qq == q)
                    sums = [None, None]
                    for rk, kv in order:
                        c = rk % nch
                        x = part[(bh, kv, q)]
                        sums[c] = x.copy() if sums[c] is None else _red_add_f32(sums[c], x)
                    want = sums[0] if nch == 1 or sums[1] is None else (sums[0] + sums[1]).astype(np.float32)
                    assert np.array_equal(got[bh, q * tile:(q + 1) * tile], want), \
                        f"{sched} (split {split}, timed {timed}), {nch} chain(s): head {bh}, dQ tile {q} differs " \
                        "from the rank-order sum"


LARGE = [w for w in workloads.WORKLOADS.values() if w.S >= 2048]


@pytest.mark.parametrize("w", LARGE, ids=[w.name for w in LARGE])
def test_full_size_sampled_heads(w):
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    heads = sorted({(0, 0), (w.B - 1, w.H - 1)})
    ref_f = P.oracle_fwd(heads)
    for (b, h), (ro, rl) in ref_f.items():
        assert_close(f"O[{b},{h}]", o[b, h], ro)
        assert err(lse[b, h], rl)[1] <= LSE_ABS_TOL
    q, k, v, do = P.f64
    ref_b = {}
    for (b, h) in heads:
        ro, rl = ref_f[(b, h)]
        sl = (slice(b, b + 1), slice(h, h + 1))
        r = A.backward(q[sl], k[sl], v[sl], ro[None, None], do[sl], rl[None, None], w.causal, P.scale)
        ref_b[(b, h)] = [x[0, 0] for x in r]
    for sched in w.schedules:
        dq, dk, dv = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, tile=w.tile)
        dash.dash_sync_status()
        for (b, h), refs in ref_b.items():
            for name, x, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
                assert_close(f"{w.name} {sched} {name}[{b},{h}]", x[b, h], r)
        # invariants on every head: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i
        dk32, dv32, do32 = dk.float(), dv.float(), P.do.float()
        scale_k = dk32.abs().amax(dim=(2, 3)) * w.S ** 0.5
        assert bool((dk32.sum(2).abs().amax(-1) <= 0.05 * scale_k + 1e-3).all())
        dvs, dos = dv32.sum(2), do32.sum(2)
        assert float((dvs - dos).norm() / dos.norm()) < 2e-2
        assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()


def test_host_buffer_entry_point_matches_device_path():
    P = Problem(1, 2, 512, 128, True)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, True, P.scale)
    dq, dk, dv = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "descending_q")
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, ho, hdo, hl = (pin(t) for t in (P.q, P.k, P.v, o, P.do, lse))
    outs = [torch.empty_like(hq).pin_memory() for _ in range(3)]
    dash.dash_attn_bwd_host(hq, hk, hv, ho, hdo, hl, *outs, True, P.scale, "descending_q")
    for a, b in zip(outs, (dq, dk, dv)):
        assert torch.equal(a, b.cpu())


@pytest.mark.parametrize("H", [5, 17])
@pytest.mark.parametrize("sched", ["shift", "serial", "atomic"])
def test_host_entry_point_in_head_groups_is_bit_identical(sched, H):
    # ten heads go through the host entry point in four groups (3 + 3 + 3 + 1);
    # thirty-four in groups of at most five (6 x 5 + 4)
    # every head's dQ order is its own, so the bits equal one device call
    # (atomic is compared within the tolerance: its order is not fixed)
    P = Problem(2, H, 512, 128, False)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, False, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, sched)
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, ho, hdo, hl = (pin(t) for t in (P.q, P.k, P.v, o, P.do, lse))
    outs = [torch.full_like(hq, float("nan")).pin_memory() for _ in range(3)]
    dash.dash_attn_bwd_host(hq, hk, hv, ho, hdo, hl, *outs, False, P.scale, sched)
    for name, a, b in zip(("dQ", "dK", "dV"), outs, ref):
        if sched == "atomic":
            assert_close(f"host {name}", a.float(), b.double().cpu().numpy(), rel=1e-3, abs_=1e-2)
        else:
            assert torch.equal(a, b.cpu()), name


def test_invalid_arguments_are_rejected():
    P = Problem(1, 2, 640, 64, True)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, True, P.scale)
    with pytest.raises(dash.DashError) as ei:   # n = 5 blocks: odd
        dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "symmetric_shift")
    assert ei.value.code == 2
    with pytest.raises(dash.DashError) as ei:
        dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "shift")
    assert ei.value.code == 2
    with pytest.raises(dash.DashError) as ei:
        dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "serial", tile=96)
    assert ei.value.code == 2
    bad = np.array([[0, 0, 9, 1 << 28 | 1 << 29]], dtype=np.int32)   # q tile out of range
    with pytest.raises(dash.DashError) as ei:
        dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "serial", tasks=bad, cta_off=[0, 1])
    assert ei.value.code == 6
