"""GPU vs oracle on small and mid-size workloads that span several tiles and
ragged tails: bit-exact index sets, diffs, runs and gathered bytes; attention
within 1e-2 abs + 1e-2 rel of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.kvo import KvoError
from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS, Workload
from tests.harness import Case, assert_attn_close
from tests.margins import MARGIN, find_attempts

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": WORKLOADS["tiny"],
    "ragged_spec": Workload("ragged_spec", 3, 8, 2, 128, 16, 24, 80, 1, (1104, 2128), spec_sigma=0.3),
    "tokens_b1": Workload("tokens_b1", 2, 8, 2, 128, 1, 300, 48, 1, (4144, 4144), plant="token_runs",
                          n_planted=300, plant_beta=12.0),
    "r8_d64_nowin": Workload("r8_d64_nowin", 2, 16, 2, 64, 32, 8, 0, 1, (2048, 2048)),
    "r16": Workload("r16", 1, 32, 2, 128, 8, 32, 32, 1, (1056, 1056), key_dist="channel_scaled"),
    "select_all": Workload("select_all", 1, 4, 1, 128, 16, 20, 16, 1, (336, 336)),
    "k1": Workload("k1", 2, 4, 2, 64, 4, 1, 8, 1, (208, 208), spec_sigma=0.5),
    "clustered": Workload("clustered", 1, 16, 2, 128, 64, 8, 64, 1, (6464, 6464), key_dist="clustered",
                          n_centroids=32, centroid_sigma=0.3),
    "multi_chunk": Workload("multi_chunk", 2, 8, 2, 128, 2, 64, 16, 1, (6016, 6016), spec_sigma=0.2),
    # 750-1500 blocks per group: six selection CTAs per group's cluster, the
    # shorter groups' last three scoring no rows
    "sel_cluster6": Workload("sel_cluster6", 3, 8, 2, 128, 4, 32, 16, 1, (3016, 6016), spec_sigma=0.3),
    # 800 register-direct tiles per group = 50 work items: more than the merge's
    # shared-memory table holds at d = 64, so the online merge runs
    "many_items": Workload("many_items", 1, 8, 2, 64, 32, 400, 32, 1, (32 + 32 * 420, 32 + 32 * 420)),
}


def _attempts(w, seed):
    lens = synth.seq_lens(w, seed)
    groups = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    if w.plant == "token_runs":
        return None
    return find_attempts(w, seed, 0, lens, lambda b, g, qr: synth.gen_request_kv(w, seed, 0, b, lens[b], qr)[0][g],
                         groups)


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    w = CASES[request.param]
    seed = 777
    c = Case(w, seed, attempts=_attempts(w, seed), gen_device="cpu")
    refs = {(b, g): c.oracle_group(0, b, g) for b in range(w.batch) for g in range(w.n_kv_heads)}
    yield c, refs
    c.close()


def test_landmarks(case):
    c, _ = case
    w = c.w
    lm = c.ctx.landmarks(0).cpu()
    for b in range(w.batch):
        for g in range(w.n_kv_heads):
            C = (c.lens[b] - w.window) // w.block_size
            ref = orc.landmarks(synth.bits(c.rows(0, b, g)), w.block_size, C)
            got = lm[b * w.n_kv_heads + g, :C].double().numpy()
            if w.block_size == 1:
                np.testing.assert_array_equal(got, ref)
            else:
                np.testing.assert_allclose(got, ref, rtol=2e-6, atol=1e-7)
            assert not lm[b * w.n_kv_heads + g, C:].any()


def test_select_topk_bit_exact(case):
    c, refs = case
    w = c.w
    T, P = c.ctx.select_topk(0, c.q_dev(0), c.q_dev(0, spec=True))
    T, P = T.cpu(), (None if P is None else P.cpu())
    for (b, g), ref in refs.items():
        assert orc.kth_relative_gap(ref.scores_true, w.top_k) >= MARGIN
        assert T[b * w.n_kv_heads + g].tolist() == ref.T.tolist(), (b, g)
        if P is not None:
            assert P[b * w.n_kv_heads + g].tolist() == ref.P.tolist(), (b, g)
    # a second call reuses the self-cleaning scratch
    T2, _ = c.ctx.select_topk(0, c.q_dev(0))
    assert torch.equal(T2.cpu(), T)
    assert c.ctx.device_status() == 0


@pytest.mark.parametrize("impl", [0, 2])
def test_select_kernels_match_the_oracle(case, impl):
    """The ticket kernel (impl 0) and the cluster kernel (impl 2, where a
    group's CTAs fit a cluster) give the oracle's indices, true and speculative."""
    c, refs = case
    w = c.w
    try:
        c.ctx.set_select_impl(impl)
        for _ in range(2):                 # the second call finds the scratch as the first left it
            T, P = c.ctx.select_topk(0, c.q_dev(0), c.q_dev(0, spec=True))
            T, P = T.cpu(), (None if P is None else P.cpu())
            for (b, g), ref in refs.items():
                assert T[b * w.n_kv_heads + g].tolist() == ref.T.tolist(), (impl, b, g)
                if P is not None:
                    assert P[b * w.n_kv_heads + g].tolist() == ref.P.tolist(), (impl, b, g)
        assert c.ctx.device_status() == 0
    finally:
        c.ctx.set_select_impl(1)


def test_select_impl_setter_checks_its_argument(case):
    c, _ = case
    for bad in (-1, 3):
        with pytest.raises(KvoError):
            c.ctx.set_select_impl(bad)


def test_diff_gather_attention_chain(case):
    c, refs = case
    w = c.w
    k, G = w.top_k, w.batch * w.n_kv_heads
    q = c.q_dev(0)
    T, P = c.ctx.select_topk(0, q, c.q_dev(0, spec=True))
    if P is None:
        P = T.clone()
    miss, cnt, slot = c.ctx.index_diff(T, P)
    runs_p, nr_p = c.ctx.gather_coalesced(0, 1, P, None, slot_base=0, urgent=False)
    runs_m, nr_m = c.ctx.gather_coalesced(0, 1, miss, cnt, slot_base=k, urgent=True)
    o, lse = c.ctx.sparse_decode_attn(0, 1, q, slot, fuse_window_merge=True)
    o2, lse2 = c.ctx.sparse_decode_attn(0, 1, q, slot, fuse_window_merge=False)
    torch.cuda.synchronize()
    assert c.ctx.device_status() == 0
    bufK, bufV = c.ctx.buffer(1)
    miss, cnt, slot = miss.cpu(), cnt.cpu(), slot.cpu()
    runs_p, nr_p, runs_m, nr_m = runs_p.cpu(), nr_p.cpu(), runs_m.cpu(), nr_m.cpu()
    bufK, bufV = synth.bits(bufK.cpu()), synth.bits(bufV.cpu())
    o, lse, o2, lse2 = o.cpu().numpy(), lse.cpu().numpy(), o2.cpu().numpy(), lse2.cpu().numpy()
    r = w.group_size
    for (b, g), ref in refs.items():
        i = b * w.n_kv_heads + g
        n_m = int(cnt[i])
        assert miss[i, :n_m].tolist() == ref.M.tolist()
        assert slot[i].tolist() == ref.slot_of_true.tolist()
        assert [tuple(x) for x in runs_p[i, :int(nr_p[i]), :3].tolist()] == ref.runs_prefetch
        assert [tuple(x) for x in runs_m[i, :int(nr_m[i]), :3].tolist()] == ref.runs_urgent
        assert not runs_p[i, :int(nr_p[i]), 3].any()
        for kv, buf in (("k", bufK), ("v", bufV)):
            exp, written = orc.gather_slots(synth.bits(c.rows(0, b, g, kv)), w.block_size,
                                            ref.runs_prefetch + ref.runs_urgent, 2 * k)
            assert np.array_equal(buf[i][written], exp[written]), (b, g, kv)
        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
        assert_attn_close(o[0, rows], ref.o)
        assert_attn_close(lse[0, rows], ref.lse, what="lse")
        assert_attn_close(o2[0, rows], ref.o_sparse, what="o_sparse")
        assert_attn_close(lse2[0, rows], ref.lse_sparse, what="lse_sparse")
        if w.window:
            assert_attn_close(o2[1, rows], ref.o_window, what="o_window")
            assert_attn_close(lse2[1, rows], ref.lse_window, what="lse_window")
        else:
            assert np.all(lse2[1, rows] == -np.inf) and not o2[1, rows].any()


@pytest.mark.parametrize("engine,drivers", [(1, 1), (1, 3), (1, 32), (2, 5), (3, 0), (4, 0)])
def test_gather_engines_bit_exact(case, engine, drivers):
    """TMA bulk copies (engines 1, 2), the flat lane-load gather (engine 3) and
    the copy engine (engine 4: one cudaMemcpyAsync per run, issued by the host)
    write the same bytes as the oracle's gather."""
    c, refs = case
    w = c.w
    k = w.top_k
    T, P = c.ctx.select_topk(0, c.q_dev(0), c.q_dev(0, spec=True))
    if P is None:
        P = T.clone()
    miss, cnt, slot = c.ctx.index_diff(T, P)
    c.ctx.set_gather_engine(engine, drivers)
    try:
        c.ctx.gather_coalesced(0, 0, P, None, slot_base=0)
        c.ctx.gather_coalesced(0, 0, miss, cnt, slot_base=k, urgent=True)
        torch.cuda.synchronize()
        assert c.ctx.device_status() == 0
    finally:
        c.ctx.set_gather_engine(3, 0)          # back to the default engine
    bufK, bufV = c.ctx.buffer(0)
    bufK, bufV = synth.bits(bufK.cpu()), synth.bits(bufV.cpu())
    for (b, g), ref in refs.items():
        i = b * w.n_kv_heads + g
        for kv, buf in (("k", bufK), ("v", bufV)):
            exp, written = orc.gather_slots(synth.bits(c.rows(0, b, g, kv)), w.block_size,
                                            ref.runs_prefetch + ref.runs_urgent, 2 * k)
            assert np.array_equal(buf[i][written], exp[written]), (b, g, kv)


def test_flat_gather_reserve_limits(case):
    """The flat gather's reservation tops out at 227 KiB less its own 128-byte
    table; the largest one still writes the oracle's bytes."""
    c, refs = case
    w = c.w
    k = w.top_k
    with pytest.raises(KvoError):
        c.ctx.set_gather_reserve(227 * 1024 - 127)
    with pytest.raises(KvoError):
        c.ctx.set_gather_reserve(-1)
    T, P = c.ctx.select_topk(0, c.q_dev(0), c.q_dev(0, spec=True))
    if P is None:
        P = T.clone()
    miss, cnt, slot = c.ctx.index_diff(T, P)
    c.ctx.set_gather_reserve(227 * 1024 - 128)
    try:
        c.ctx.gather_coalesced(0, 1, P, None, slot_base=0)
        c.ctx.gather_coalesced(0, 1, miss, cnt, slot_base=k, urgent=True)
        torch.cuda.synchronize()
        assert c.ctx.device_status() == 0
    finally:
        c.ctx.set_gather_reserve(200 * 1024)
    bufK, bufV = c.ctx.buffer(1)
    bufK, bufV = synth.bits(bufK.cpu()), synth.bits(bufV.cpu())
    for (b, g), ref in refs.items():
        i = b * w.n_kv_heads + g
        for kv, buf in (("k", bufK), ("v", bufV)):
            exp, written = orc.gather_slots(synth.bits(c.rows(0, b, g, kv)), w.block_size,
                                            ref.runs_prefetch + ref.runs_urgent, 2 * k)
            assert np.array_equal(buf[i][written], exp[written]), (b, g, kv)


@pytest.mark.parametrize("ctas", [0, 1, 3])
def test_attention_kernels_agree(case, ctas):
    """The register-direct kernel (impl 0) and the TMA-staged persistent kernel
    (impl 1; ctas > 0 gives each CTA a longer tile range, several work items
    and stage-ring reuse across them) both match the oracle.  They split the
    tiles differently, so they agree to rounding, not bit for bit."""
    c, refs = case
    w = c.w
    r = w.group_size
    q = c.q_dev(0)
    qs = c.q_dev(0, spec=True)
    T, _ = c.ctx.select_topk(0, q)
    miss, cnt, slot = c.ctx.index_diff(T, None)
    c.ctx.gather_coalesced(0, 0, miss, cnt, slot_base=w.top_k, urgent=True)
    out = {}
    try:
        for impl in (0, 1):
            c.ctx.set_attn_impl(impl, ctas if impl == 1 else 0)
            res = [t.cpu() for t in c.ctx.sparse_decode_attn(0, 0, q, slot, fuse_window_merge=True)]
            res += [t.cpu() for t in c.ctx.sparse_decode_attn(0, 0, q, slot, fuse_window_merge=False)]
            if qs is not None and 2 * r <= 16:
                res += [t.cpu() for t in c.ctx.sparse_decode_attn_cobatch(0, 0, q, qs, slot)]
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            out[impl] = res
    finally:
        c.ctx.set_attn_impl(2, 0)
    for a, b in zip(out[0], out[1]):
        assert a.shape == b.shape
        np.testing.assert_allclose(b.numpy(), a.numpy(), rtol=1e-2, atol=2e-3)
    for impl in (0, 1):
        o, lse, o2, lse2 = (t.numpy() for t in out[impl][:4])
        for (b, g), ref in refs.items():
            rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
            assert_attn_close(o[0, rows], ref.o)
            assert_attn_close(lse[0, rows], ref.lse, what="lse")
            assert_attn_close(o2[0, rows], ref.o_sparse, what="o_sparse")
            assert_attn_close(lse2[0, rows], ref.lse_sparse, what="lse_sparse")
            if w.window:
                assert_attn_close(o2[1, rows], ref.o_window, what="o_window")
                assert_attn_close(lse2[1, rows], ref.lse_window, what="lse_window")


@pytest.mark.parametrize("per_group", [0, 1, 3, 8])
def test_cluster_attention_matches_oracle(case, per_group):
    """The group-split cluster kernel (impl 2): per_group CTAs per group (0: as
    many as fill the device; 3 leaves uneven shares that cut a part inside a
    CTA; 8 on the small cases gives CTAs with no tiles at all) attend with one
    softmax over both parts and merge through distributed shared memory.  The
    fused output, the co-batched output and -- through the persistent kernel it
    falls back to -- the separate parts all match the oracle."""
    c, refs = case
    w = c.w
    r = w.group_size
    q = c.q_dev(0)
    qs = c.q_dev(0, spec=True)
    if qs is None:
        qs = (q.float() * 0.5).to(torch.bfloat16)     # any second query works
    T, _ = c.ctx.select_topk(0, q)
    miss, cnt, slot = c.ctx.index_diff(T, None)
    c.ctx.gather_coalesced(0, 0, miss, cnt, slot_base=w.top_k, urgent=True)
    try:
        c.ctx.set_attn_impl(2, per_group)
        o, lse = (t.cpu().numpy() for t in c.ctx.sparse_decode_attn(0, 0, q, slot, fuse_window_merge=True))
        o2, lse2 = (t.cpu().numpy() for t in c.ctx.sparse_decode_attn(0, 0, q, slot, fuse_window_merge=False))
        cob = None
        if 2 * r <= 16:
            cob = [t.cpu().numpy() for t in c.ctx.sparse_decode_attn_cobatch(0, 0, q, qs, slot)]
        torch.cuda.synchronize()
        assert c.ctx.device_status() == 0
    finally:
        c.ctx.set_attn_impl(2, 0)
    qs_bits = synth.bits(qs.cpu()) if cob is not None else None
    for (b, g), ref in refs.items():
        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
        assert_attn_close(o[0, rows], ref.o)
        assert_attn_close(lse[0, rows], ref.lse, what="lse")
        assert_attn_close(o2[0, rows], ref.o_sparse, what="o_sparse")
        assert_attn_close(lse2[0, rows], ref.lse_sparse, what="lse_sparse")
        if w.window:
            assert_attn_close(o2[1, rows], ref.o_window, what="o_window")
            assert_attn_close(lse2[1, rows], ref.lse_window, what="lse_window")
        if cob is not None:
            assert_attn_close(cob[0][0, rows], ref.o, what="cobatched o")
            rs = orc.decode_group(synth.bits(c.rows(0, b, g, "k")), synth.bits(c.rows(0, b, g, "v")),
                                  synth.bits(c.q[0][b, g * r:(g + 1) * r]), qs_bits[b, g * r:(g + 1) * r],
                                  block_size=w.block_size, top_k=w.top_k, window=w.window)
            assert_attn_close(cob[2][0, rows], rs.o_spec, what="cobatched o_spec")
            assert_attn_close(cob[3][0, rows], rs.lse_spec, what="cobatched lse_spec")


def test_cobatched_attention(case):
    """True and speculative queries in one attention pass (2r <= 16)."""
    c, refs = case
    w = c.w
    if 2 * w.group_size > 16:
        pytest.skip("co-batching needs 2r <= 16")
    q = c.q_dev(0)
    qs = c.q_dev(0, spec=True)
    if qs is None:
        qs = (q.float() * 0.5).to(torch.bfloat16)     # any second query works
    T, _ = c.ctx.select_topk(0, q)
    miss, cnt, slot = c.ctx.index_diff(T, None)
    c.ctx.gather_coalesced(0, 0, miss, cnt, slot_base=w.top_k, urgent=True)
    o1, l1 = c.ctx.sparse_decode_attn(0, 0, q, slot)
    o2, l2 = c.ctx.sparse_decode_attn(0, 0, qs, slot)
    o, lse, os_, ls_ = c.ctx.sparse_decode_attn_cobatch(0, 0, q, qs, slot)
    torch.cuda.synchronize()
    assert c.ctx.device_status() == 0
    np.testing.assert_allclose(o.cpu().numpy(), o1.cpu().numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(os_.cpu().numpy(), o2.cpu().numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(ls_.cpu().numpy(), l2.cpu().numpy(), rtol=1e-5, atol=1e-5)
    r = w.group_size
    qs_bits = synth.bits(qs.cpu())
    for (b, g), ref in refs.items():
        rr = orc.decode_group(synth.bits(c.rows(0, b, g, "k")), synth.bits(c.rows(0, b, g, "v")),
                              synth.bits(c.q[0][b, g * r:(g + 1) * r]), qs_bits[b, g * r:(g + 1) * r],
                              block_size=w.block_size, top_k=w.top_k, window=w.window)
        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
        assert_attn_close(os_[0, rows].cpu().numpy(), rr.o_spec, what="o_spec")
        assert_attn_close(ls_[0, rows].cpu().numpy(), rr.lse_spec, what="lse_spec")


def test_merge_lse_matches_fused(case):
    from sparse_kv_cache_landmark_gb300.kvo import merge_lse
    c, refs = case
    w = c.w
    q = c.q_dev(0)
    T, _ = c.ctx.select_topk(0, q)
    miss, cnt, slot = c.ctx.index_diff(T, None)
    c.ctx.gather_coalesced(0, 0, miss, cnt, slot_base=w.top_k, urgent=True)
    o, lse = c.ctx.sparse_decode_attn(0, 0, q, slot, fuse_window_merge=True)
    parts, lparts = c.ctx.sparse_decode_attn(0, 0, q, slot, fuse_window_merge=False)
    om, lm = merge_lse(parts[0], lparts[0], parts[1], lparts[1])
    torch.cuda.synchronize()
    np.testing.assert_allclose(om.cpu().numpy(), o[0].cpu().numpy(), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(lm.cpu().numpy(), lse[0].cpu().numpy(), rtol=1e-5, atol=1e-5)
    r = w.group_size
    for (b, g), ref in refs.items():
        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
        assert_attn_close(om[rows].cpu().numpy(), ref.o)


def test_generator_is_device_independent():
    w = CASES["ragged_spec"]
    lens = synth.seq_lens(w, 5)
    q, _ = synth.gen_queries(w, 5, 0)
    for b in range(w.batch):
        Kc, Vc = synth.gen_request_kv(w, 5, 0, b, lens[b], q[b], device="cpu")
        Kg, Vg = synth.gen_request_kv(w, 5, 0, b, lens[b], q[b], device="cuda")
        assert torch.equal(Kc.view(torch.int16), Kg.cpu().view(torch.int16))
        assert torch.equal(Vc.view(torch.int16), Vg.cpu().view(torch.int16))
    wt = WORKLOADS["tiny"]
    qt, _ = synth.gen_queries(wt, 5, 0)
    Kc, _ = synth.gen_request_kv(wt, 5, 0, 0, 4096, qt[0], device="cpu")
    Kg, _ = synth.gen_request_kv(wt, 5, 0, 0, 4096, qt[0], device="cuda")
    assert torch.equal(Kc.view(torch.int16), Kg.cpu().view(torch.int16))


def test_merge_lse_edge_cases():
    from sparse_kv_cache_landmark_gb300.kvo import merge_lse
    d = 8
    o1 = torch.randn(4, d, device="cuda")
    o2 = torch.randn(4, d, device="cuda")
    l1 = torch.tensor([0.5, -float("inf"), -float("inf"), 3.0], device="cuda")
    l2 = torch.tensor([-float("inf"), 1.0, -float("inf"), 3.0], device="cuda")
    o, lse = merge_lse(o1, l1, o2, l2)
    o, lse = o.cpu(), lse.cpu()
    assert torch.allclose(o[0], o1[0].cpu()) and lse[0] == 0.5
    assert torch.allclose(o[1], o2[1].cpu()) and lse[1] == 1.0
    assert not o[2].any() and lse[2] == -float("inf")
    exp, el = orc.merge_lse(o1[3].cpu().double().numpy(), 3.0, o2[3].cpu().double().numpy(), 3.0)
    np.testing.assert_allclose(o[3].numpy(), exp, rtol=1e-5, atol=1e-6)
    assert abs(float(lse[3]) - el) < 1e-5


def test_bad_index_lists_set_the_status_word():
    w = CASES["r8_d64_nowin"]
    c = Case(w, 3, gen_device="cpu")
    try:
        G, k = w.batch * w.n_kv_heads, w.top_k
        C = (c.lens[0] - w.window) // w.block_size
        # out-of-range ids: flagged, never used as addresses
        bad = torch.full((G, k), C + 5, dtype=torch.int32, device="cuda")
        c.ctx.index_diff(bad, None)
        assert c.ctx.device_status() & 1
        c.ctx.gather_coalesced(0, 0, bad, None, slot_base=0)
        # the flat engine rejects the ids themselves, the run-walking engines the runs past C_b
        assert c.ctx.device_status() & (1 | 2)
        c.ctx.set_gather_engine(0, 0)
        c.ctx.gather_coalesced(0, 0, bad, None, slot_base=0)
        assert c.ctx.device_status() & 2
        c.ctx.set_gather_engine(3, 0)
        # descending ids: flagged as unsorted
        desc = torch.arange(k - 1, -1, -1, dtype=torch.int32, device="cuda").repeat(G, 1).contiguous()
        c.ctx.index_diff(desc, None)
        assert c.ctx.device_status() & 8
        # counts outside [0, k]
        good = torch.arange(k, dtype=torch.int32, device="cuda").repeat(G, 1).contiguous()
        cnt = torch.full((G,), k + 3, dtype=torch.int32, device="cuda")
        c.ctx.gather_coalesced(0, 0, good, cnt, slot_base=0)
        assert c.ctx.device_status() & 4
        assert c.ctx.device_status() == 0
    finally:
        c.close()
