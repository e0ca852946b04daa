"""Pins of the fp64 oracle against things other than itself: hand-derived
fixtures, closed forms, brute force on tiny inputs, library routines on special
cases and structural invariants.  CPU only."""
import json
import math
import os
import struct

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _ev(x):
    if isinstance(x, str):
        return eval(x, {"__builtins__": {}}, {"e": math.e, "log": math.log, "sqrt": math.sqrt})
    if isinstance(x, list):
        return [_ev(v) for v in x]
    return x


def _bits(values):
    """bf16 bit patterns of values that are exact in bf16 (small integers here)."""
    out = []
    for v in np.asarray(values, dtype=np.float64).reshape(-1):
        u = struct.unpack("<I", struct.pack("<f", float(v)))[0]
        assert u & 0xFFFF == 0, "fixture value not exact in bf16"
        out.append(u >> 16)
    return np.array(out, dtype=np.uint16).reshape(np.shape(values))


# --------------------------------------------------------------------- format
def test_bf16_upcast_known_patterns():
    got = orc.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x3EAA, 0x0000, 0x8000, 0x7F7F], dtype=np.uint16))
    assert got[0] == 1.0 and got[1] == -2.0
    assert got[2] == 0.33203125
    assert got[3] == 0.0 and math.copysign(1.0, got[4]) == -1.0
    assert got[5] == float.fromhex("0x1.fep127")


def test_group_tokens_ragged_layout():
    # 2 requests (lens 3 and 2), 2 KV heads, d = 2; element value encodes (b, g, t, c)
    lens, H, d = [3, 2], 2, 2
    flat = []
    for b, n in enumerate(lens):
        for g in range(H):
            for t in range(n):
                for c in range(d):
                    flat.append(1000 * b + 100 * g + 10 * t + c)
    flat = np.array(flat)
    rows = orc.group_tokens(flat, lens, H, d, 1, 1)
    assert rows.tolist() == [[1100, 1101], [1110, 1111]]
    rows = orc.group_tokens(flat, lens, H, d, 0, 1)
    assert rows[:, 0].tolist() == [100, 110, 120]


# ------------------------------------------------------------------ landmarks
def test_landmarks_constant_keys_closed_form():
    B, C, d = 4, 5, 3
    keys = np.repeat(np.arange(C * d, dtype=np.float64).reshape(C, 1, d) - 7.0, B, axis=1).reshape(C * B, d)
    lm = orc.landmarks(_bits(keys), B, C)
    np.testing.assert_array_equal(lm, keys.reshape(C, B, d)[:, 0, :])


def test_landmarks_brute_force_loops():
    rng = np.random.default_rng(0)
    B, C, d = 3, 4, 2
    vals = rng.integers(-8, 8, size=(C * B + 2, d)).astype(np.float64)   # 2 trailing window rows ignored
    lm = orc.landmarks(_bits(vals), B, C)
    for j in range(C):
        for c in range(d):
            s = 0.0
            for t in range(B):
                s += vals[j * B + t, c]
            assert lm[j, c] == s / B


def test_landmark_block1_is_key():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**15, size=(9, 4)).astype(np.uint16) & 0x3FFF
    lm = orc.landmarks(bits, 1, 9)
    np.testing.assert_array_equal(lm, orc.bf16_bits_to_f64(bits))


# ------------------------------------------------------------------- scoring
def test_scores_sum_over_group_heads():
    lm = np.array([[1.0, 0, 0], [0, 1.0, 0], [0, 0, 1.0], [1.0, 1.0, 1.0]])
    q = _bits([[1.0, 2.0, 0.0], [0.0, -4.0, 8.0]])      # u = [1, -2, 8]
    np.testing.assert_array_equal(orc.block_scores(q, lm), [1.0, -2.0, 8.0, 7.0])


# --------------------------------------------------------------------- top-k
def test_topk_hand_cases():
    for case in _load("topk_cases.json")["cases"]:
        got = orc.topk_blocks(np.array(case["scores"]), case["k"])
        assert got.tolist() == case["expected"], case


def test_topk_matches_full_sort_and_margin():
    rng = np.random.default_rng(2)
    for _ in range(20):
        n = int(rng.integers(5, 300))
        k = int(rng.integers(1, n + 1))
        s = rng.standard_normal(n)
        ref = np.sort(np.argsort(-s, kind="stable")[:k])
        assert orc.topk_blocks(s, k).tolist() == ref.tolist()
        gap = orc.kth_relative_gap(s, k)
        srt = np.sort(s)[::-1]
        if k < n:
            assert gap == pytest.approx((srt[k - 1] - srt[k]) / abs(srt[k - 1]))
        else:
            assert gap == math.inf


# ---------------------------------------------------------------- diff / runs
def test_diff_and_runs_hand_cases():
    fx = _load("diff_runs_cases.json")
    for c in fx["diff_cases"]:
        M, slot = orc.index_diff(c["T"], c["P"], c["k"])
        assert M.tolist() == c["M"] and slot.tolist() == c["slot_of_true"], c
    for c in fx["run_cases"]:
        assert [list(r) for r in orc.coalesce_runs(c["S"], c["base"])] == c["runs"], c


def test_diff_invariants_random():
    rng = np.random.default_rng(3)
    for _ in range(50):
        n = int(rng.integers(2, 200))
        k = int(rng.integers(1, n + 1))
        T = np.sort(rng.choice(n, k, replace=False))
        P = np.sort(rng.choice(n, k, replace=False))
        M, slot = orc.index_diff(T, P, k)
        assert len(M) == len(set(P.tolist()) - set(T.tolist()))
        assert M.tolist() == sorted(set(T.tolist()) - set(P.tolist()))
        for i, t in enumerate(T):
            if slot[i] < k:
                assert P[slot[i]] == t
            else:
                assert M[slot[i] - k] == t
        assert len(set(slot.tolist())) == k
        M2, slot2 = orc.index_diff(T, T, k)
        assert len(M2) == 0 and slot2.tolist() == list(range(k))


def test_runs_invariants_random():
    rng = np.random.default_rng(4)
    for _ in range(50):
        n = int(rng.integers(1, 300))
        S = np.sort(rng.choice(400, n, replace=False))
        runs = orc.coalesce_runs(S, 7)
        rebuilt = [x for (s, L, _) in runs for x in range(s, s + L)]
        assert rebuilt == S.tolist()
        assert len(runs) == 1 + int(np.sum(np.diff(S) != 1))
        assert [r[2] for r in runs] == [7 + int(np.searchsorted(S, r[0])) for r in runs]


def test_gather_slots_copies_host_bytes():
    rng = np.random.default_rng(5)
    B, d, n_blk = 3, 4, 10
    rows = rng.integers(0, 65535, size=(n_blk * B, d)).astype(np.uint16)
    runs = orc.coalesce_runs([1, 2, 6], 0) + orc.coalesce_runs([8], 3)
    buf, written = orc.gather_slots(rows, B, runs, 6)
    assert written.tolist() == [True, True, True, True, False, False]
    for slot, blk in [(0, 1), (1, 2), (2, 6), (3, 8)]:
        assert buf[slot].tobytes() == rows[blk * B:(blk + 1) * B].tobytes()


# ----------------------------------------------------------------- attention
def test_attention_two_token_fixture():
    fx = _load("attention_two_token.json")
    o, lse = orc.attention_part(np.array(_ev(fx["q"])), np.array(fx["K"], float), np.array(fx["V"], float))
    np.testing.assert_allclose(o, fx["expected_o"], rtol=0, atol=1e-14)
    assert lse == pytest.approx(_ev(fx["expected_lse"]), abs=1e-14)


def test_attention_single_token_and_uniform_keys():
    rng = np.random.default_rng(6)
    d = 8
    q, k, v = rng.standard_normal(d), rng.standard_normal((1, d)), rng.standard_normal((1, d))
    o, lse = orc.attention_part(q, k, v)
    np.testing.assert_allclose(o, v[0], atol=1e-15)
    assert lse == pytest.approx(float(q @ k[0]) / math.sqrt(d), abs=1e-14)
    n = 7
    K = np.repeat(k, n, axis=0)
    V = rng.standard_normal((n, d))
    o, lse = orc.attention_part(q, K, V)
    np.testing.assert_allclose(o, V.mean(axis=0), atol=1e-14)
    assert lse == pytest.approx(float(q @ k[0]) / math.sqrt(d) + math.log(n), abs=1e-13)


def test_attention_matches_scipy_softmax():
    rng = np.random.default_rng(7)
    d, n = 16, 50
    q, K, V = rng.standard_normal(d), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    z = K @ q / math.sqrt(d)
    o, lse = orc.attention_part(q, K, V)
    np.testing.assert_allclose(o, softmax(z) @ V, atol=1e-13)
    assert lse == pytest.approx(logsumexp(z), abs=1e-12)


def test_merge_identity_disjoint_halves():
    rng = np.random.default_rng(8)
    d, n = 16, 40
    for cut in [1, 13, 39]:
        q, K, V = rng.standard_normal(d) * 2, rng.standard_normal((n, d)), rng.standard_normal((n, d))
        o1, l1 = orc.attention_part(q, K[:cut], V[:cut])
        o2, l2 = orc.attention_part(q, K[cut:], V[cut:])
        o, lse = orc.merge_lse(o1, l1, o2, l2)
        z = K @ q / math.sqrt(d)
        np.testing.assert_allclose(o, softmax(z) @ V, atol=1e-12)
        assert lse == pytest.approx(logsumexp(z), abs=1e-12)
    o, lse = orc.merge_lse(np.ones(d), 0.5, np.zeros(d), -math.inf)
    np.testing.assert_array_equal(o, np.ones(d))
    assert lse == 0.5
    o, lse = orc.merge_lse(np.zeros(d), -math.inf, np.zeros(d), -math.inf)
    assert lse == -math.inf and not o.any()


# ------------------------------------------------------------ whole pipeline
def test_hand_pipeline_fixture():
    fx = _load("hand_pipeline.json")
    sh, E = fx["shape"], fx["expected"]
    res = orc.decode_group(_bits(fx["K"]), _bits(fx["V"]), _bits(fx["q"]), _bits(fx["q_spec"]),
                           block_size=sh["block_size"], top_k=sh["top_k"], window=sh["window"])
    lm = orc.landmarks(_bits(fx["K"]), sh["block_size"], 4)
    np.testing.assert_array_equal(lm, E["landmarks"])
    np.testing.assert_array_equal(res.scores_true, E["scores_true"])
    np.testing.assert_array_equal(res.scores_pred, E["scores_pred"])
    assert res.T.tolist() == E["T"] and res.P.tolist() == E["P"] and res.M.tolist() == E["M"]
    assert res.slot_of_true.tolist() == E["slot_of_true"]
    assert [list(r) for r in res.runs_prefetch] == E["runs_prefetch"]
    assert [list(r) for r in res.runs_urgent] == E["runs_urgent"]
    np.testing.assert_allclose(res.o_sparse, _ev(E["o_sparse"]), atol=1e-14)
    np.testing.assert_allclose(res.lse_sparse, _ev(E["lse_sparse"]), atol=1e-14)
    np.testing.assert_allclose(res.o_window, E["o_window"], atol=1e-14)
    np.testing.assert_allclose(res.lse_window, _ev(E["lse_window"]), atol=1e-14)
    np.testing.assert_allclose(res.o, _ev(E["o"]), atol=1e-14)
    np.testing.assert_allclose(res.lse, _ev(E["lse"]), atol=1e-14)


def test_all_blocks_selected_equals_dense_attention():
    rng = np.random.default_rng(9)
    B, C, W, d, r = 4, 6, 5, 8, 3
    n = C * B + W
    K = rng.integers(-20, 20, size=(n, d)) / 8.0
    V = rng.integers(-20, 20, size=(n, d)) / 8.0
    q = rng.integers(-20, 20, size=(r, d)) / 8.0
    res = orc.decode_group(_bits(K), _bits(V), _bits(q), None, block_size=B, top_k=C, window=W)
    assert res.T.tolist() == list(range(C)) and len(res.M) == 0
    for h in range(r):
        z = K @ q[h] / math.sqrt(d)
        np.testing.assert_allclose(res.o[h], softmax(z) @ V, atol=1e-12)
        assert res.lse[h] == pytest.approx(logsumexp(z), abs=1e-12)


def test_prediction_never_changes_output():
    # DualDecoder core claim: after urgent correction, attention equals the
    # ground-truth sparse selection, whatever the prediction was.
    rng = np.random.default_rng(10)
    B, C, W, d, r, k = 2, 12, 4, 8, 2, 4
    n = C * B + W
    K = rng.integers(-20, 20, size=(n, d)) / 8.0
    V = rng.integers(-20, 20, size=(n, d)) / 8.0
    q = rng.integers(-20, 20, size=(r, d)) / 8.0
    base = orc.decode_group(_bits(K), _bits(V), _bits(q), None, block_size=B, top_k=k, window=W)
    for pred in ([], [0, 1, 2, 3], base.T.tolist(), [8, 9, 10, 11]):
        res = orc.decode_group(_bits(K), _bits(V), _bits(q), None, block_size=B, top_k=k, window=W,
                               prediction=pred)
        assert res.T.tolist() == base.T.tolist()
        np.testing.assert_array_equal(res.o, base.o)
        assert len(res.M) == len(set(base.T.tolist()) - set(pred))


def test_cobatched_speculative_rows():
    # the speculative query attends to the true selection plus the window
    rng = np.random.default_rng(11)
    B, C, W, d, r, k = 2, 10, 3, 8, 2, 4
    n = C * B + W
    K = rng.integers(-20, 20, size=(n, d)) / 8.0
    V = rng.integers(-20, 20, size=(n, d)) / 8.0
    q = rng.integers(-20, 20, size=(r, d)) / 8.0
    qs = rng.integers(-20, 20, size=(r, d)) / 8.0
    res = orc.decode_group(_bits(K), _bits(V), _bits(q), _bits(qs), block_size=B, top_k=k, window=W)
    toks = np.concatenate([np.arange(x * B, (x + 1) * B) for x in res.T] + [np.arange(n - W, n)])
    for h in range(r):
        z = K[toks] @ qs[h] / math.sqrt(d)
        np.testing.assert_allclose(res.o_spec[h], softmax(z) @ V[toks], atol=1e-12)
        assert res.lse_spec[h] == pytest.approx(logsumexp(z), abs=1e-12)
    same = orc.decode_group(_bits(K), _bits(V), _bits(q), _bits(q), block_size=B, top_k=k, window=W)
    np.testing.assert_array_equal(same.o_spec, same.o)
    assert orc.decode_group(_bits(K), _bits(V), _bits(q), None, block_size=B, top_k=k, window=W).o_spec is None
