"""Cross-step delta prefetch (resident block sets, kv_offload_init resident = 1)
against the oracle over several decode steps with drifting queries: the slot
tables and the fetch counts are bit-exact, attention is within the tolerance,
and every occupied slot holds its block's bytes."""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close
from tests.margins import MARGIN

pytestmark = pytest.mark.gpu


def _attempts(c, steps, drift):
    """Per layer, attempts [b][Hkv] giving every group its selection margin at every step."""
    w = c.w
    r = w.group_size
    out = []
    for l in range(c.L):
        a = np.zeros((w.batch, w.n_kv_heads), dtype=np.int64)
        for b in range(w.batch):
            for g in range(w.n_kv_heads):
                C = (c.lens[b] - w.window) // w.block_size
                lm = orc.landmarks(synth.bits(c.rows(l, b, g)), w.block_size, C)
                for att in range(300):
                    ok = True
                    for s in range(steps):
                        qg, qsg = synth.gen_group_query_step(w, c.seed, l, b, g, s, drift, att)
                        gaps = [orc.kth_relative_gap(orc.block_scores(synth.bits(qg), lm), w.top_k)]
                        if qsg is not None:
                            gaps.append(orc.kth_relative_gap(orc.block_scores(synth.bits(qsg), lm), w.top_k))
                        if min(gaps) < MARGIN:
                            ok = False
                            break
                    if ok:
                        a[b, g] = att
                        break
                else:
                    raise AssertionError("no attempt with margins at every step")
        out.append(a)
    return out


@pytest.mark.parametrize("spec,L,B,k,dual,budget,W,ragged,graphs", [
    (True, 2, 16, 16, True, None, 32, False, False), (False, 1, 16, 16, False, None, 32, False, False),
    (True, 1, 1, 64, False, None, 32, False, False), (True, 3, 32, 8, False, None, 32, False, False),
    (True, 2, 16, 16, False, 3, 32, False, False),
    (True, 1, 16, 16, False, None, 0, False, False),   # no window: attention over the resident blocks alone
    (True, 2, 32, 12, False, None, 64, True, False),   # ragged lengths, k not a multiple of the warp count
    (False, 2, 32, 12, False, None, 64, True, False),  # no speculation: one chain, every SM copies the misses
    (False, 2, 32, 12, False, None, 64, True, True),   # ... replayed from CUDA graphs
    ("alt", 2, 16, 16, False, None, 32, False, False),  # speculative and plain steps alternate
    ("s3", 2, 16, 16, False, None, 32, False, True),   # graph replays, one speculative step, replays again
    (False, 1, 16, 8, False, None, 32, "many", False),  # 320 groups: one CTA per group for the fetched blocks
    (False, 2, 32, 12, False, None, 64, True, "impl0"),  # chain steps with the register-direct attention
    (False, 2, 32, 12, False, None, 64, True, "impl2g"),  # chain steps, group-split cluster attention, graphs
    (False, 2, 1, 24, False, None, 32, True, "sel2"),  # B = 1: 600-640 blocks, three selection CTAs per cluster
    (False, 2, 1, 24, False, None, 32, True, "sel0"),  # ... with the ticket selection kernel
    (True, 2, 16, 16, True, None, 32, False, "impl2")])  # speculative resident steps, cluster attention
def test_resident_steps_match_the_oracle(spec, L, B, k, dual, budget, W, ragged, graphs):
    drift, steps, seed = 0.15, 6, 321
    n = W + B * 64 if B > 1 else W + 600
    if ragged == "many":
        w = Workload(f"resident_B{B}_many", 40, 16, 8, 128, B, k, W, L, (n, n), spec_sigma=None)
        ragged, graphs, steps = False, False, 3
    else:
        ctx = (n, n + 40 * B) if ragged else (n, n)
        w = Workload(f"resident_B{B}", 3 if ragged else 2, 8, 2, 128, B, k, W, L, ctx,
                     spec_sigma=0.3 if spec else None)
    c = Case(w, seed, gen_device="cpu", resident=True)
    try:
        att = _attempts(c, steps, drift)
        if budget is not None:
            c.ctx.set_prefetch_budget(budget)     # admission cap on speculative fetches
        if graphs in ("sel0", "sel2"):
            # the fused assignment in the ticket kernel's last CTA / the cluster's first CTA
            c.ctx.set_select_impl(0 if graphs == "sel0" else 2)
            graphs = False
        elif graphs == "impl0":
            c.ctx.set_attn_impl(0)                # one attention pass after the copy, whole set
            graphs = False
        elif graphs in ("impl2", "impl2g"):
            c.ctx.set_attn_impl(2, 2)             # two CTAs per group: the clusters merge in shared memory
            graphs = graphs == "impl2g"
        if graphs:
            c.ctx.set_graphs(True)
        G, r = w.batch * w.n_kv_heads, w.group_size
        state = [[[-1] * (2 * k) for _ in range(G)] for _ in range(L)]
        p_cur = [[None] * G for _ in range(L)]
        n_urg = n_pref = 0
        churn = []
        for s in range(steps):
            spec_s = spec is True or (spec == "alt" and s % 2 == 0) or (spec == "s3" and s == 3)
            qq = [synth.gen_queries_step(w, seed, l, s, drift, att[l]) for l in range(L)]
            q = torch.stack([x[0] for x in qq]).cuda().contiguous()
            qs = torch.stack([x[1] for x in qq]).cuda().contiguous() if spec_s else None
            if graphs:
                # the same q, o and lse buffers every step, so warm chain steps replay one graph per parity
                if s == 0:
                    q_buf = torch.empty_like(q)
                    o_buf = torch.empty(L, w.batch * w.n_q_heads, w.head_dim, dtype=torch.float32, device="cuda")
                    lse_buf = torch.empty(L, w.batch * w.n_q_heads, dtype=torch.float32, device="cuda")
                q_buf.copy_(q)
                o_buf.fill_(float("nan"))
                o, lse = c.ctx.decode_step(q_buf, qs, o_buf, lse_buf)
            elif dual:
                o, lse, o_sp, lse_sp = c.ctx.decode_step_dual(q, qs)
            else:
                o, lse = c.ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            o, lse = o.cpu().numpy(), lse.cpu().numpy()
            fetched_step = 0
            for l in range(L):
                table = c.ctx.resident_slots(l).numpy()
                for b in range(w.batch):
                    for g in range(w.n_kv_heads):
                        i = b * w.n_kv_heads + g
                        qg = synth.bits(qq[l][0][b, g * r:(g + 1) * r])
                        qsg = synth.bits(qq[l][1][b, g * r:(g + 1) * r]) if spec_s else None
                        ref = orc.decode_group(synth.bits(c.rows(l, b, g, "k")), synth.bits(c.rows(l, b, g, "v")),
                                               qg, qsg, block_size=B, top_k=k, window=W)
                        new, urg, _, pref = orc.resident_step(state[l][i], ref.T.tolist(), p_cur[l][i],
                                                              ref.P.tolist() if spec_s else None, budget)
                        state[l][i] = new
                        p_cur[l][i] = ref.P.tolist() if spec_s else ref.T.tolist()
                        n_urg += len(urg)
                        n_pref += len(pref)
                        fetched_step += len(urg) + len(pref)
                        assert table[i].tolist() == new, (s, l, b, g)
                        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                        assert_attn_close(o[l, rows], ref.o, what=f"o step {s} layer {l}")
                        assert_attn_close(lse[l, rows], ref.lse, what=f"lse step {s} layer {l}")
                        if dual:
                            assert_attn_close(o_sp[l, rows].cpu().numpy(), ref.o_spec, what="o_spec")
            churn.append(fetched_step)
            assert c.ctx.resident_fetched() == (n_urg, n_pref)
        # the first step fetches everything; later steps only the drift's delta
        assert churn[0] >= L * G * k and max(churn[1:]) < churn[0]
        # every occupied slot holds its block's bytes
        for l in range(L):
            bk, bv = c.ctx.buffer(2 + l)
            bk, bv = synth.bits(bk.cpu()), synth.bits(bv.cpu())
            for b in range(w.batch):
                for g in range(w.n_kv_heads):
                    i = b * w.n_kv_heads + g
                    kr, vr = synth.bits(c.rows(l, b, g, "k")), synth.bits(c.rows(l, b, g, "v"))
                    for sl, x in enumerate(state[l][i]):
                        if x >= 0:
                            assert np.array_equal(bk[i, sl], kr[x * B:(x + 1) * B])
                            assert np.array_equal(bv[i, sl], vr[x * B:(x + 1) * B])
    finally:
        c.close()


def test_resident_setters_check_their_arguments():
    w = Workload("res_args", 1, 4, 1, 64, 16, 4, 16, 1, (16 + 16 * 8, 16 + 16 * 8))
    c = Case(w, 1, gen_device="cpu", resident=True)
    try:
        with pytest.raises(Exception, match="blocks"):
            c.ctx.set_prefetch_budget(-2)
        c.ctx.set_prefetch_budget(-1)
        with pytest.raises(Exception, match="layer"):
            c.ctx.resident_slots(1)
        with pytest.raises(Exception, match="implementation"):
            c.ctx.set_attn_impl(3)
        with pytest.raises(Exception, match="implementation"):
            c.ctx.set_attn_impl(2, 9)
        with pytest.raises(Exception, match="implementation"):
            c.ctx.set_attn_impl(1, -1)
        c.ctx.set_attn_impl(2, 0)
    finally:
        c.close()


def test_resident_calls_need_resident_mode():
    w = Workload("plain", 1, 4, 1, 64, 16, 4, 16, 1, (16 + 16 * 8, 16 + 16 * 8))
    c = Case(w, 1, gen_device="cpu")
    try:
        with pytest.raises(Exception, match="resident"):
            c.ctx.resident_slots(0)
        with pytest.raises(Exception, match="resident"):
            c.ctx.resident_fetched()
        with pytest.raises(Exception, match="resident"):
            c.ctx.set_prefetch_budget(4)
    finally:
        c.close()


def test_adaptive_speculation_stops_when_prefetches_do_not_pay():
    """With a speculative query that predicts badly (noise 1.0), prefetching
    every step's prediction moves more host bytes than fetching only the
    misses.  The adaptive policy counts, per layer, how many prefetched blocks
    a later true index used and stops prefetching a layer whose prefetches are
    used less than half the time, so it must recover most of that waste --
    while every output still matches the oracle (the true index is always
    completed by urgent fetches)."""
    steps, drift, seed = 24, 0.15, 77
    n = 32 + 16 * 64
    w = Workload("spec_policy", 2, 8, 2, 128, 16, 16, 32, 2, (n, n), spec_sigma=1.0)
    r, G = w.group_size, w.batch * w.n_kv_heads
    totals, final = {}, {}
    for mode in ("always", "adaptive", "none"):
        c = Case(w, seed, gen_device="cpu", resident=True)
        try:
            if mode == "adaptive":
                c.ctx.set_spec_policy(1)
            # the last step's true query gets its selection margin (its outputs are compared)
            att = []
            for l in range(w.n_layers):
                a = np.zeros((w.batch, w.n_kv_heads), dtype=np.int64)
                for b in range(w.batch):
                    for g in range(w.n_kv_heads):
                        C = (c.lens[b] - w.window) // w.block_size
                        lm = orc.landmarks(synth.bits(c.rows(l, b, g)), w.block_size, C)
                        for t in range(300):
                            qg, _ = synth.gen_group_query_step(w, seed, l, b, g, steps - 1, drift, t)
                            if orc.kth_relative_gap(orc.block_scores(synth.bits(qg), lm), w.top_k) >= MARGIN:
                                a[b, g] = t
                                break
                        else:
                            raise AssertionError("no attempt with a margin")
                att.append(a)
            for s in range(steps):
                qq = [synth.gen_queries_step(w, seed, l, s, drift, att[l]) for l in range(w.n_layers)]
                q = torch.stack([x[0] for x in qq]).cuda().contiguous()
                qs = None if mode == "none" else torch.stack([x[1] for x in qq]).cuda().contiguous()
                o, lse = c.ctx.decode_step(q, qs)
                torch.cuda.synchronize()
                assert c.ctx.device_status() == 0
            totals[mode] = sum(c.ctx.resident_fetched())
            if mode != "none":
                final[mode] = c.ctx.spec_stats()
            o, lse = o.cpu().numpy(), lse.cpu().numpy()
            for l in range(w.n_layers):
                for b in range(w.batch):
                    for g in range(w.n_kv_heads):
                        qg = synth.bits(qq[l][0][b, g * r:(g + 1) * r])
                        ref = orc.decode_group(synth.bits(c.rows(l, b, g, "k")), synth.bits(c.rows(l, b, g, "v")),
                                               qg, None, block_size=w.block_size, top_k=w.top_k, window=w.window)
                        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                        assert_attn_close(o[l, rows], ref.o, what=f"o {mode} layer {l}")
                        assert_attn_close(lse[l, rows], ref.lse, what=f"lse {mode} layer {l}")
        finally:
            c.close()
    # bad predictions: always prefetching costs host bytes; the counters say so
    assert totals["always"] > totals["none"]
    for pf, used, _ in final["always"]:
        assert pf > 0 and 2 * used < pf
    # the adaptive policy recovers most of the waste
    waste = totals["always"] - totals["none"]
    assert totals["adaptive"] <= totals["none"] + 0.6 * waste, totals
    assert any(on == 0 for *_, on in final["adaptive"]) or totals["adaptive"] < totals["always"]
