"""Oracle on the synthetic workloads: the planted structure is recovered and
the selection margins hold (CPU)."""
import numpy as np

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS
from tests.margins import MARGIN, find_attempts


def _krows_fn(w, seed, lens):
    def k_rows(b, g, q_req):
        K, _ = synth.gen_request_kv(w, seed, 0, b, lens[b], q_req)
        return K[g]
    return k_rows


def test_tiny_planted_blocks_selected_with_margin():
    w, seed = WORKLOADS["tiny"], 1234
    lens = synth.seq_lens(w, seed)
    groups = [(0, g) for g in range(w.n_kv_heads)]
    att = find_attempts(w, seed, 0, lens, _krows_fn(w, seed, lens), groups)
    L = synth.make_layer(w, seed, attempts=att)
    res = orc.decode_layer(synth.bits(L.k), synth.bits(L.v), synth.bits(L.q), None, L.lens,
                           n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
                           top_k=w.top_k, window=w.window)
    for (b, g), r in res.items():
        planted = synth.planted_blocks(w, seed, 0, b, g, 252).tolist()
        assert set(planted) <= set(r.T.tolist())
        assert orc.kth_relative_gap(r.scores_true, w.top_k) >= MARGIN
        assert len(r.T) == w.top_k and len(r.M) == 0


def test_fragmentation_group_recovers_planted_runs():
    full = WORKLOADS["fragmentation"]
    w = full.scaled(batch=1, n_q_heads=full.group_size, n_kv_heads=1)    # group (0, 0) of the full shape
    seed = 1238
    L = synth.make_layer(w, seed)
    res = orc.decode_layer(synth.bits(L.k), synth.bits(L.v), synth.bits(L.q), None, L.lens,
                           n_kv_heads=1, head_dim=w.head_dim, block_size=1, top_k=w.top_k,
                           window=w.window)[(0, 0)]
    planted = synth.planted_blocks(w, seed, 0, 0, 0, 65024).tolist()
    assert res.T.tolist() == planted
    assert orc.kth_relative_gap(res.scores_true, w.top_k) > 0.1
    n_iso = sum(1 for (_, n, _) in res.runs_prefetch if n == 1)
    assert n_iso == round(0.6 * 2048)
    assert all(n <= 64 for (_, n, _) in res.runs_prefetch)


def test_long_context_prediction_overlap_near_88_percent():
    full = WORKLOADS["long_ctx_predict"]
    w = full.scaled(batch=6, n_q_heads=full.group_size, n_kv_heads=1)
    seed = 99
    lens = synth.seq_lens(w, seed)
    q, qs = synth.gen_queries(w, seed, 0)
    ov = []
    for b in range(w.batch):
        K, _ = synth.gen_request_kv(w, seed, 0, b, lens[b], q[b])
        lm = orc.landmarks(synth.bits(K[0]), w.block_size, (lens[b] - w.window) // w.block_size)
        T = orc.topk_blocks(orc.block_scores(synth.bits(q[b]), lm), w.top_k)
        P = orc.topk_blocks(orc.block_scores(synth.bits(qs[b]), lm), w.top_k)
        M, slot = orc.index_diff(T, P, w.top_k)
        ov.append(1 - len(M) / w.top_k)
    assert 0.82 < np.mean(ov) < 0.94, ov
