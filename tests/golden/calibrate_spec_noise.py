"""Calibrate the speculative-query noise of the long-context workload.

DualDecoder (abstract; Fig. 16) reports that the retrieval index predicted from
the speculative token overlaps the true one by 88% on average.  This script
finds the sigma of q_spec = q + sigma * N(0,1) that gives a mean overlap
|T n P| / k of 0.88 on the long-context workload's shapes, using only the
seeded generator and the oracle's scoring / top-k.  Its output is the constant
SPEC_SIGMA_88 in sparse_kv_cache_landmark_gb300/workloads.py.

    python tests/golden/calibrate_spec_noise.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import oracle as orc  # noqa: E402
from sparse_kv_cache_landmark_gb300 import synth  # noqa: E402
from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS  # noqa: E402


def main(n_req=16, seed=4321):
    full = WORKLOADS["long_ctx_predict"]
    # one KV head per request (r = 4 as in the full shape): same streams as group (b, 0)
    w = full.scaled(batch=n_req, n_q_heads=full.group_size, n_kv_heads=1, spec_sigma=1.0)
    lens = synth.seq_lens(w, seed)
    q, e1 = synth.gen_queries(w, seed, 0)           # q_spec at sigma = 1 -> noise = q_spec - q
    lms = []
    for b in range(n_req):
        K, _ = synth.gen_request_kv(w, seed, 0, b, lens[b], q[b])
        C = (lens[b] - w.window) // w.block_size
        lms.append(orc.landmarks(synth.bits(K[0]), w.block_size, C))
    qf = q.float()
    noise = (e1.float() - qf)          # bf16(q + e) - q, close to e; only used to search sigma
    import torch

    def overlap(sig):
        ov = []
        for b in range(n_req):
            qs = (qf[b] + sig * noise[b]).to(torch.bfloat16)
            T = orc.topk_blocks(orc.block_scores(synth.bits(q[b]), lms[b]), w.top_k)
            P = orc.topk_blocks(orc.block_scores(synth.bits(qs), lms[b]), w.top_k)
            ov.append(len(set(T.tolist()) & set(P.tolist())) / w.top_k)
        return float(np.mean(ov))

    lo, hi = 0.0, 1.0
    for _ in range(14):
        mid = 0.5 * (lo + hi)
        if overlap(mid) > 0.88:
            lo = mid
        else:
            hi = mid
    sig = round(0.5 * (lo + hi), 3)
    # check with the generator's own formula q_spec = bf16(q + sigma * e)
    _, qs = synth.gen_queries(w.scaled(spec_sigma=sig), seed, 0)
    ov = []
    for b in range(n_req):
        T = orc.topk_blocks(orc.block_scores(synth.bits(q[b]), lms[b]), w.top_k)
        P = orc.topk_blocks(orc.block_scores(synth.bits(qs[b]), lms[b]), w.top_k)
        ov.append(len(set(T.tolist()) & set(P.tolist())) / w.top_k)
    print(f"sigma={sig} search-overlap={overlap(sig):.4f} generator-overlap={np.mean(ov):.4f}")


if __name__ == "__main__":
    main()
