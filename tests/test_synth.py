"""The seeded generator: hash, distributions and planted structure (CPU)."""
import numpy as np
import torch

from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS


def test_mix32_tensor_matches_int():
    rng = np.random.default_rng(0)
    xs = rng.integers(0, 2**32, size=1000, dtype=np.uint64).astype(np.int64)
    got = synth.mix32(torch.from_numpy(xs)).numpy()
    assert [synth.mix32_int(int(x)) for x in xs] == got.tolist()
    assert synth.mix32_int(0) == 0 and synth.mix32_int(1) != 1


def test_normal_table_is_a_symmetric_monotone_unit_normal():
    t = synth.normal_table_bits().astype(np.uint32) << np.uint32(16)
    v = t.view(np.float32).astype(np.float64)
    assert np.all(np.diff(v) >= 0)
    np.testing.assert_array_equal(v, -v[::-1])
    assert abs(v.mean()) < 1e-6 and abs(v.std() - 1.0) < 2e-3


def test_queries_are_deterministic_and_attempts_reseed():
    w = WORKLOADS["long_ctx_predict"].scaled(batch=2)
    q1, s1 = synth.gen_queries(w, 7, 0)
    q2, s2 = synth.gen_queries(w, 7, 0)
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    a = np.zeros((2, 8), dtype=np.int64); a[1, 3] = 5
    q3, _ = synth.gen_queries(w, 7, 0, a)
    r = w.group_size
    diff = (q3.view(torch.int16) != q1.view(torch.int16)).any(dim=-1)
    assert diff[1, 3 * r:4 * r].all() and diff.sum() == r
    # speculative noise is small
    assert (s1.float() - q1.float()).std() < 0.2


def test_seq_lens_ranges():
    w = WORKLOADS["long_ctx_predict"]
    lens = synth.seq_lens(w, 1236)
    assert all(65536 <= n <= 131072 and n % 32 == 0 for n in lens)
    assert len(set(lens)) > 50
    assert synth.seq_lens(WORKLOADS["llama3_8b_decode"], 1) == [32768] * 16


def test_token_runs_structure():
    w = WORKLOADS["fragmentation"]
    ids = synth.planted_blocks(w, 11, 0, 3, 5, 65024).numpy()
    assert len(ids) == 2048 and len(set(ids.tolist())) == 2048 and ids.max() < 65024 and ids.min() >= 0
    runs = []
    for x in ids.tolist():
        if runs and x == runs[-1][0] + runs[-1][1]:
            runs[-1][1] += 1
        else:
            runs.append([x, 1])
    lens = [L for _, L in runs]
    assert sum(1 for L in lens if L == 1) == round(0.6 * 2048)
    assert all(2 <= L <= 64 for L in lens if L > 1)


def test_planted_blocks_distinct():
    w = WORKLOADS["tiny"]
    ids = synth.planted_blocks(w, 1, 0, 0, 1, 252).numpy()
    assert len(ids) == 8 and len(set(ids.tolist())) == 8 and np.all(np.diff(ids) > 0)


def test_channel_scale_and_clusters():
    w = WORKLOADS["llama3_8b_decode"].scaled(batch=1)
    q, _ = synth.gen_queries(w, 3, 0)
    K, V = synth.gen_request_kv(w, 3, 0, 0, 2048, q[0])
    std_c = K[0].float().std(dim=0)
    assert std_c.min() > 0.35 and std_c.max() < 2.3 and std_c.max() / std_c.min() > 2.0
    wc = WORKLOADS["wide_budget"].scaled(batch=1)
    q, _ = synth.gen_queries(wc, 3, 0)
    K, _ = synth.gen_request_kv(wc, 3, 0, 0, 64 * 40, q[0])
    blk = K[0].float().view(40, 64, 128)
    # tokens of one block scatter around one centroid with sigma ~0.3
    assert 0.2 < (blk - blk.mean(dim=1, keepdim=True)).std() < 0.4


def test_step_queries_reduce_to_single_step_and_drift_as_stated():
    from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS
    w = WORKLOADS["long_ctx_predict"].scaled(batch=2)
    q0, qs0 = synth.gen_queries(w, 5, 0)
    q, qs = synth.gen_queries_step(w, 5, 0, 0, 0.0)
    assert torch.equal(q, q0) and torch.equal(qs, qs0)
    # q_s - q_0(drift 0) ~ drift * N(0,1); q_spec_s - q_{s+1} ~ sigma * N(0,1)
    drift = 0.1
    qa, qsa = synth.gen_queries_step(w, 5, 0, 3, drift)
    qb, _ = synth.gen_queries_step(w, 5, 0, 4, drift)
    assert abs((qa.float() - q0.float()).std().item() - drift) < 0.01
    assert abs((qsa.float() - qb.float()).std().item() - w.spec_sigma) < 0.01
    # without speculation there is no q_spec; steps differ only through the drift
    w2 = WORKLOADS["llama3_8b_decode"].scaled(batch=1)
    qc, qsc = synth.gen_queries_step(w2, 5, 0, 2, 0.0)
    assert qsc is None and torch.equal(qc, synth.gen_queries(w2, 5, 0)[0])
