"""Plain fp64 CPU oracle of one sparse offloaded-KV decode step (per layer).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py``; never by the product library.
Single-threaded numpy, float64 throughout, no blocking or fusion beyond the
definitions below.  Every function names the passage it follows:

* "DualDecoder: Accelerate Long Context LLM Inference by Predictive Prefetch"
  (arXiv 2607.26475) -- §4.1 / Fig. 6 / Fig. 8: the retrieval index of a step
  is computed from a (true or speculative) token and static GPU-resident K
  landmarks; §5.2 / Fig. 10 / Fig. 18: entries missing from the prediction are
  fetched on an urgent stream before attention; §5.4 / Fig. 11: two-layer
  ping-pong sparse KV buffer; Fig. 19: contiguous block prefetch, then a GPU
  reorder; core claim: attention over the miss-corrected buffer equals
  attention over the ground-truth sparse selection.
* "PulseInfer and the I/O Problem Behind Long-Context Decoding", §2: a
  gather-scatter I/O engine that coalesces fragmented transfers.
* "Scaling Attention Beyond GPUs for LLM Inference" (abstract): dense
  attention over the recent entries plus sparse attention over salient
  entries, fused through a log-sum-exp scheme.

The pages give no formula; where a step is left open the plainest reading is
taken and stated in the docstring (landmark = mean key of a block; per-KV-head
score = sum over the GQA group of q_h . landmark; exact top-k with ties to the
lower block id; misses placed after the k prefetch slots; coalescing by exact
adjacency only; softmax scale 1/sqrt(d), natural-log lse).

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
brute force, closed forms, identities and hand-computed fixtures in
``tests/golden/``.

Layouts (all arrays are numpy):
* bf16 values travel as their 16-bit patterns (``uint16``/``int16``);
* host K/V of one layer are packed ``[b][Hkv][len_b][d]`` request after request;
* q is ``[b][Hq][d]``; KV head g serves query heads ``g*r .. g*r+r-1``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "group_tokens", "landmarks", "block_scores", "topk_blocks",
    "kth_relative_gap", "index_diff", "coalesce_runs", "gather_slots", "resident_assign", "resident_step",
    "lowrank_keys", "f32_to_bf16_bits",
    "attention_part", "merge_lse", "GroupResult", "decode_group", "decode_layer",
]


# ----------------------------------------------------------------------------
# number format
# ----------------------------------------------------------------------------
def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact bf16 -> float64: a bf16 value is the top half of an IEEE float32."""
    u16 = np.asarray(bits).astype(np.uint16)
    f32 = (u16.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return f32.astype(np.float64)


def group_tokens(kv_packed, seq_lens, n_kv_heads: int, head_dim: int, b: int, g: int) -> np.ndarray:
    """Token rows ``[len_b][d]`` of request b, KV head g, from a packed layer array."""
    flat = np.asarray(kv_packed).reshape(-1)
    start = int(sum(int(x) for x in seq_lens[:b])) * n_kv_heads * head_dim
    n = int(seq_lens[b])
    off = start + g * n * head_dim
    return flat[off: off + n * head_dim].reshape(n, head_dim)


# ----------------------------------------------------------------------------
# step 1: landmarks and block scores   (DualDecoder §4.1, Fig. 6, Fig. 8)
# ----------------------------------------------------------------------------
def landmarks(k_rows_bits, block_size: int, n_blocks: int) -> np.ndarray:
    """K landmark of block j = mean of the keys of tokens [j*B, (j+1)*B).

    Reading: the pages name "K landmarks" kept on the GPU (DualDecoder §4.1,
    Fig. 8) in the QUEST/ShadowKV style without a formula; the mean key per
    block is taken.  For B = 1 the landmark is the key itself.
    Returns float64 ``[n_blocks][d]``.
    """
    K = bf16_bits_to_f64(k_rows_bits)[: n_blocks * block_size]
    d = K.shape[1]
    out = np.zeros((n_blocks, d))
    for j in range(n_blocks):
        out[j] = K[j * block_size:(j + 1) * block_size].sum(axis=0) / block_size
    return out


def block_scores(q_group_bits, lm: np.ndarray) -> np.ndarray:
    """Per-KV-head score of every candidate block (DualDecoder §4.1).

    s_j = sum over the r query heads h of the group of  q_h . L_j
    (no softmax, no 1/sqrt(d): neither changes the ranking).
    """
    Q = bf16_bits_to_f64(q_group_bits)            # [r][d]
    return np.einsum("hc,jc->j", Q, lm)


def topk_blocks(scores: np.ndarray, k: int) -> np.ndarray:
    """Retrieval index: the k highest-scoring blocks, emitted in ascending id order.

    Exact selection: order blocks by (score descending, id ascending) and keep
    the first k, so equal scores go to the lower block id.
    """
    n = scores.shape[0]
    k = min(k, n)
    order = sorted(range(n), key=lambda j: (-scores[j], j))
    return np.array(sorted(order[:k]), dtype=np.int64)


def kth_relative_gap(scores: np.ndarray, k: int) -> float:
    """(s_(k) - s_(k+1)) / |s_(k)| for the k-th and (k+1)-th largest scores (inf if k >= n)."""
    n = scores.shape[0]
    if k >= n or k <= 0:
        return math.inf
    s = np.sort(scores)[::-1]
    denom = abs(s[k - 1])
    return math.inf if denom == 0.0 else float((s[k - 1] - s[k]) / denom)


# ----------------------------------------------------------------------------
# step 2: predicted-vs-needed diff   (DualDecoder §5.2, Fig. 10, Fig. 18)
# ----------------------------------------------------------------------------
def index_diff(T, P, k: int):
    """Misses and slot map of the true index T against the prediction P.

    M = T minus P (ascending): the entries the urgent stream must fetch.
    slot_of_true[i] = position of T[i] in P if predicted (already prefetched into
    slot pos), else k + rank of T[i] in M (reading: misses go to their own slot
    range after the k prefetch slots, so each destination stays contiguous).
    """
    T = [int(x) for x in T]
    P = [int(x) for x in P]
    pos_in_P = {x: i for i, x in enumerate(P)}
    M = [x for x in T if x not in pos_in_P]
    rank_in_M = {x: i for i, x in enumerate(M)}
    slot = [pos_in_P[x] if x in pos_in_P else k + rank_in_M[x] for x in T]
    return np.array(M, dtype=np.int64), np.array(slot, dtype=np.int64)


# ----------------------------------------------------------------------------
# step 3: coalesced gather   (PulseInfer §2; DualDecoder Fig. 1, Fig. 19)
# ----------------------------------------------------------------------------
def coalesce_runs(S, slot_base: int):
    """Maximal runs of consecutive block ids in the ascending list S.

    A run starts at i = 0 and wherever S[i] != S[i-1] + 1.  Each run is
    (first block id, number of blocks, destination slot = slot_base + i) in list
    order.  Reading: exact adjacency only, no gap filling, no length cap.
    """
    runs = []
    for i, x in enumerate(int(v) for v in S):
        if runs and x == runs[-1][0] + runs[-1][1]:
            runs[-1][1] += 1
        else:
            runs.append([x, 1, slot_base + i])
    return [tuple(r) for r in runs]


def gather_slots(rows_bits, block_size: int, runs, n_slots: int):
    """Buffer content the runs produce: slot s holds the B token rows of its block.

    Returns (buffer ``[n_slots][B][d]`` of bit patterns, written mask ``[n_slots]``).
    """
    rows = np.asarray(rows_bits)
    d = rows.shape[1]
    buf = np.zeros((n_slots, block_size, d), dtype=rows.dtype)
    written = np.zeros(n_slots, dtype=bool)
    for first, n, dst in runs:
        for m in range(n):
            blk = first + m
            buf[dst + m] = rows[blk * block_size:(blk + 1) * block_size]
            written[dst + m] = True
    return buf, written


# ----------------------------------------------------------------------------
# cross-step residency: delta prefetch
#   ("NeuroPrefetcher: Storage-Aware Sparse LLM Inference via Delta
#   Prefetching", title: fetch only what the previous step did not bring;
#   DualDecoder §5.2 / Fig. 18: misses of the true index are fetched urgently)
# ----------------------------------------------------------------------------
def resident_assign(slots, need, keep=None, budget=None):
    """Make every block of ``need`` resident in one (layer, group)'s slot table.

    ``slots``: sequence of length cap, the block id held by each slot (-1:
    empty).  ``need``: ascending block ids that must be resident afterwards.
    ``keep``: ascending block ids (or None) whose slots must not be reused.

    Reading (the pages name delta prefetching but give no rule): blocks of
    ``need`` already resident stay in their slots; the missing ones, in
    ascending id order, take the reusable slots in ascending slot order, a slot
    being reusable when it is empty or holds a block in neither ``need`` nor
    ``keep``.

    ``budget`` (None: no limit) admits at most that many fetches: the missing
    blocks with the lowest ids are fetched, the rest stay out (an admission cap
    on host bytes; "PulseInfer and the I/O Problem Behind Long-Context
    Decoding", §2 names I/O-adaptive offloading admission without a rule).

    Returns (new slot table as a list, fetched [(block id, slot)] in ascending
    id order, slot of each entry of ``need``, -1 for entries left out by the
    budget).  Raises ValueError when the reusable slots are too few.
    """
    new = [int(x) for x in slots]
    where = {b: s for s, b in enumerate(new) if b >= 0}
    need = [int(x) for x in need]
    protect = set(need) | (set(int(x) for x in keep) if keep is not None else set())
    missing = [x for x in need if x not in where]
    if budget is not None:
        missing = missing[:max(0, int(budget))]
    reusable = [s for s, b in enumerate(new) if b < 0 or b not in protect]
    if len(missing) > len(reusable):
        raise ValueError("not enough reusable slots")
    fetched = []
    for x, s in zip(missing, reusable):
        new[s] = x
        fetched.append((x, s))
    where = {b: s for s, b in enumerate(new) if b >= 0}
    return new, fetched, [where.get(x, -1) for x in need]


def resident_step(slots, T, P_cur, P_next, budget=None):
    """One decode step of one (layer, group) with a resident block set.

    Urgent phase: the true index T becomes resident, sparing the blocks of the
    prediction P_cur made one step earlier (None on a cold start).  Prefetch
    phase (after attention): the prediction P_next for the next step becomes
    resident, sparing the blocks of T.  With a slot table of 2k entries neither
    phase runs out of slots (k blocks needed, at most k more protected).

    ``budget`` caps the prefetch phase's fetches (the urgent phase is never
    capped: the true index must be resident for attention).

    Returns (table after both phases, urgent fetches, slot of each T entry,
    prefetch fetches); with P_next None the prefetch phase is skipped.
    """
    slots, urgent, slot_of_true = resident_assign(slots, T, P_cur)
    pref = []
    if P_next is not None:
        slots, pref, _ = resident_assign(slots, P_next, T, budget)
    return slots, urgent, slot_of_true, pref


# ----------------------------------------------------------------------------
# low-rank key reconstruction   (DualDecoder §5.3: keys of missed entries are
# rebuilt on the GPU from a GPU-resident low-rank key cache instead of fetched)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def lowrank_keys(coef_bits, basis_bits) -> np.ndarray:
    """Key rows of rank-R factors as the synthetic low-rank keys define them.

    K[t][c] = bf16( sum over j = 0 .. R-1 ascending of a[t][j] * e[j][c] ), with
    a ``[n][R]`` and e ``[R][d]`` bf16, every product and every partial sum
    rounded to float32 (no fused multiply-add), the total rounded to bf16 to
    nearest-even.  Returns uint16 bits ``[n][d]``.  The precision is the one the
    keys are defined with, so this is their exact value, not an approximation.
    """
    a = bf16_bits_to_f64(coef_bits).astype(np.float32)
    e = bf16_bits_to_f64(basis_bits).astype(np.float32)
    acc = np.zeros((a.shape[0], e.shape[1]), dtype=np.float32)
    for j in range(a.shape[1]):
        prod = (a[:, j:j + 1] * e[j:j + 1, :]).astype(np.float32)
        acc = (acc + prod).astype(np.float32)
    return f32_to_bf16_bits(acc)


# ----------------------------------------------------------------------------
# step 4: attention parts and their log-sum-exp merge
#         ("Scaling Attention Beyond GPUs for LLM Inference", abstract)
# ----------------------------------------------------------------------------
def attention_part(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Softmax attention of one query over a key set; returns (o, lse).

    z_t = q.K_t / sqrt(d);  m = max z;  l = sum exp(z_t - m);
    o = sum exp(z_t - m) V_t / l;  lse = m + ln l.  An empty set gives (0, -inf).
    """
    d = q.shape[0]
    if K.shape[0] == 0:
        return np.zeros(d), -math.inf
    z = (K @ q) / math.sqrt(d)
    m = float(z.max())
    p = np.exp(z - m)
    ell = float(p.sum())
    o = (p @ V) / ell
    return o, m + math.log(ell)


def merge_lse(o1, lse1: float, o2, lse2: float):
    """Fuse two attention parts over disjoint key sets by their log-sum-exp.

    M = max(lse1, lse2); w_i = exp(lse_i - M); o = (w1 o1 + w2 o2)/(w1 + w2);
    lse = M + ln(w1 + w2).  Two empty parts give (0, -inf).
    """
    o1 = np.asarray(o1, dtype=np.float64)
    o2 = np.asarray(o2, dtype=np.float64)
    M = max(lse1, lse2)
    if M == -math.inf:
        return np.zeros_like(o1), -math.inf
    w1 = math.exp(lse1 - M)
    w2 = math.exp(lse2 - M)
    return (w1 * o1 + w2 * o2) / (w1 + w2), M + math.log(w1 + w2)


# ----------------------------------------------------------------------------
# one (request, KV head) group through all four steps
# ----------------------------------------------------------------------------
@dataclass
class GroupResult:
    T: np.ndarray                      # true retrieval index, ascending
    P: np.ndarray                      # predicted index (== T without a speculative query)
    scores_true: np.ndarray
    scores_pred: np.ndarray
    M: np.ndarray                      # misses, ascending
    slot_of_true: np.ndarray
    runs_prefetch: list
    runs_urgent: list
    o_sparse: np.ndarray               # [r][d]
    lse_sparse: np.ndarray             # [r]
    o_window: np.ndarray
    lse_window: np.ndarray
    o: np.ndarray                      # merged
    lse: np.ndarray
    o_spec: np.ndarray = None          # speculative query over the same key set (co-batched)
    lse_spec: np.ndarray = None
    extra: dict = field(default_factory=dict)


def decode_group(k_rows_bits, v_rows_bits, q_group_bits, q_spec_group_bits, *,
                 block_size: int, top_k: int, window: int, prediction=None) -> GroupResult:
    """Steps 1-4 for one (request b, KV head g) with len_b = rows.

    ``prediction`` (ascending ids) is the index predicted in an earlier step; when
    None it is computed here from ``q_spec_group_bits`` (the dual-token scheme of
    DualDecoder §5.2) or equals T when no speculative query is given.
    """
    n_tok = np.asarray(k_rows_bits).shape[0]
    C = (n_tok - window) // block_size                 # host-resident candidate blocks
    lm = landmarks(k_rows_bits, block_size, C)
    s_true = block_scores(q_group_bits, lm)
    T = topk_blocks(s_true, top_k)
    if q_spec_group_bits is not None:
        s_pred = block_scores(q_spec_group_bits, lm)
        P_new = topk_blocks(s_pred, top_k)
    else:
        s_pred = s_true
        P_new = T
    P = P_new if prediction is None else np.asarray(prediction, dtype=np.int64)
    M, slot = index_diff(T, P, top_k)
    runs_p = coalesce_runs(P, 0)
    runs_m = coalesce_runs(M, top_k)

    K = bf16_bits_to_f64(k_rows_bits)
    V = bf16_bits_to_f64(v_rows_bits)
    Q = bf16_bits_to_f64(q_group_bits)
    sel = np.concatenate([np.arange(x * block_size, (x + 1) * block_size) for x in T]) \
        if len(T) else np.zeros(0, dtype=np.int64)
    win = np.arange(n_tok - window, n_tok)
    r, d = Q.shape
    o_s = np.zeros((r, d)); l_s = np.zeros(r)
    o_w = np.zeros((r, d)); l_w = np.zeros(r)
    o = np.zeros((r, d)); lse = np.zeros(r)
    for h in range(r):
        o_s[h], l_s[h] = attention_part(Q[h], K[sel], V[sel])
        o_w[h], l_w[h] = attention_part(Q[h], K[win], V[win])
        o[h], lse[h] = merge_lse(o_s[h], l_s[h], o_w[h], l_w[h])
    # Co-batched speculative rows (DualDecoder §5.2, Fig. 18: the real and the
    # speculative token attend in one batched pass).  Reading: the speculative
    # query attends to the same key set as the true one (the true selection plus
    # the window), each part merged by log-sum-exp like the true query's.
    o_sp = l_sp = None
    if q_spec_group_bits is not None:
        Qs = bf16_bits_to_f64(q_spec_group_bits)
        o_sp = np.zeros((r, d)); l_sp = np.zeros(r)
        for h in range(r):
            a = attention_part(Qs[h], K[sel], V[sel])
            b_ = attention_part(Qs[h], K[win], V[win])
            o_sp[h], l_sp[h] = merge_lse(a[0], a[1], b_[0], b_[1])
    return GroupResult(T=T, P=P, scores_true=s_true, scores_pred=s_pred, M=M, slot_of_true=slot,
                       runs_prefetch=runs_p, runs_urgent=runs_m, o_sparse=o_s, lse_sparse=l_s,
                       o_window=o_w, lse_window=l_w, o=o, lse=lse, o_spec=o_sp, lse_spec=l_sp)


def decode_layer(k_packed, v_packed, q_bits, q_spec_bits, seq_lens, *, n_kv_heads: int,
                 head_dim: int, block_size: int, top_k: int, window: int, groups=None):
    """decode_group over every (b, g) of one layer (or the listed ``groups``)."""
    q_bits = np.asarray(q_bits)
    b_n, hq, d = q_bits.shape
    r = hq // n_kv_heads
    if groups is None:
        groups = [(b, g) for b in range(b_n) for g in range(n_kv_heads)]
    out = {}
    for b, g in groups:
        kr = group_tokens(k_packed, seq_lens, n_kv_heads, head_dim, b, g)
        vr = group_tokens(v_packed, seq_lens, n_kv_heads, head_dim, b, g)
        qg = q_bits[b, g * r:(g + 1) * r]
        qs = None if q_spec_bits is None else np.asarray(q_spec_bits)[b, g * r:(g + 1) * r]
        out[(b, g)] = decode_group(kr, vr, qg, qs, block_size=block_size, top_k=top_k,
                                   window=window)
    return out
