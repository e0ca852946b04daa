"""Selection-margin helper for the tests (uses the oracle).

The fp32 GPU scores and the fp64 oracle scores pick the same index set when
the k-th and (k+1)-th scores of a group differ by at least 1e-3 relative.  The
generator re-seeds a group's query (``attempts[b, g]``) until its margin holds,
for the true and the speculative query alike.
"""
import numpy as np
import torch

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth

MARGIN = 1e-3


def group_margin(w, lm, qg, qsg):
    gaps = [orc.kth_relative_gap(orc.block_scores(synth.bits(qg), lm), w.top_k)]
    if qsg is not None:
        gaps.append(orc.kth_relative_gap(orc.block_scores(synth.bits(qsg), lm), w.top_k))
    return min(gaps)


def find_attempts(w, seed, layer, lens, k_rows, groups, max_attempts=400):
    """attempts ``[b][Hkv]`` (zeros outside ``groups``) giving every listed group the margin.

    ``k_rows(b, g, q_request)`` returns the group's key rows (bf16 tensor
    ``[len_b][d]``); it is called again per attempt only for planted workloads,
    whose planted keys follow the query.
    """
    att = np.zeros((w.batch, w.n_kv_heads), dtype=np.int64)
    r = w.group_size
    for b, g in groups:
        C = (lens[b] - w.window) // w.block_size
        lm = None
        for a in range(max_attempts):
            qg, qsg = synth.gen_group_query(w, seed, layer, b, g, a)
            if lm is None or w.plant is not None:
                q_req = torch.zeros(w.n_q_heads, w.head_dim, dtype=torch.bfloat16)
                q_req[g * r:(g + 1) * r] = qg
                lm = orc.landmarks(synth.bits(k_rows(b, g, q_req)), w.block_size, C)
            if group_margin(w, lm, qg, qsg) >= MARGIN:
                att[b, g] = a
                break
        else:
            raise RuntimeError(f"no attempt within {max_attempts} gives group {(b, g)} the margin")
    return att
