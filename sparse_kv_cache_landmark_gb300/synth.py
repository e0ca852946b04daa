"""Seeded synthetic inputs for the sparse offloaded-KV decode step.

This module only makes inputs (queries, host K/V caches, lengths); it holds
none of the decode step's arithmetic.  It is shared by the tests, the CUDA
path's harness and the oracle, and gives bit-identical bf16 values on any
torch device: every draw is a counter-based integer hash (Chris Wellons'
"lowbias32" mixer, applied twice) evaluated with exact int64 tensor ops, and
the only float steps are single IEEE fp32 multiplies/adds rounded to bf16.

Distributions
* N(0,1): 16 hash bits index a table of the 65536 normal quantiles
  Phi^-1((u + 0.5) / 65536) rounded to bf16 (tails clipped at +-4.32).
* U(0,1): 24 hash bits / 2^24.

Recipe per workload (see ``workloads.py``)
* q, V ~ N(0,1); K ~ N(0,1), or N(0,1) * s_c with a per-(layer, KV head,
  channel) scale s_c ~ U(0.5, 2) ("channel_scaled"), or mu_m + sigma N(0,1) with
  one of 32 per-(request, KV head) centroids mu_m ~ N(0,1) drawn per block
  ("clustered"), or a rank-R product ("lowrank"): K[t][c] = bf16(sum_j
  a[t][j] * e[j][c]) with bf16 coefficients a ~ N(0,1) and basis rows
  e ~ N(0,1)/sqrt(R), the sum taken in ascending j with every multiply and add
  rounded to fp32 (so a GPU that repeats those roundings rebuilds K exactly).
* planting: the keys of chosen blocks / tokens get + beta * u_hat, u_hat the
  unit direction of the group's summed query, so they are high scorers.
  "token_runs" places 60% of the planted tokens as isolated tokens and 40% in
  runs of U{2..64}, every segment separated by at least one unplanted token.
* speculative query: q_spec = q + sigma * N(0,1) (sigma set per workload).
* decode steps (cross-step runs): step s has q_s = n + delta * e_s and
  q_spec_s = n + delta * e_{s+1} + sigma * f_s, with n, e_s, f_s ~ N(0,1)
  drawn per step, so the speculative query is a noisy draw of the next step's
  query; step 0 with delta = 0 is the single-step draw above.
* ``attempts[b, g]`` re-seeds the query streams of one (request, KV head) group,
  so a caller can redraw a group whose selection margin is too thin.
"""
from __future__ import annotations

import math
import statistics
from typing import Dict, List, Optional

import numpy as np
import torch

from .workloads import Workload

MASK32 = 0xFFFFFFFF

# stream ids
_Q, _QS, _K, _V, _KS, _MU, _ASSIGN, _PLANT, _LEN, _SEG, _QD, _LRC, _LRB = range(1, 14)


# ---------------------------------------------------------------------------
# hashing
# ---------------------------------------------------------------------------
def mix32_int(x: int) -> int:
    """lowbias32 on a Python int (mod 2^32)."""
    x &= MASK32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & MASK32
    x ^= x >> 15
    x = (x * 0x846CA68B) & MASK32
    x ^= x >> 16
    return x


def _mul32(t: torch.Tensor, c: int) -> torch.Tensor:
    # (t * c) mod 2^32 for 0 <= t < 2^32 without leaving int64's range
    lo = (t & 0xFFFF) * c
    hi = ((t >> 16) * c) & 0xFFFF
    return (lo + (hi << 16)) & MASK32


def mix32(t: torch.Tensor) -> torch.Tensor:
    """lowbias32 on an int64 tensor holding values in [0, 2^32)."""
    t = t ^ (t >> 16)
    t = _mul32(t, 0x7FEB352D)
    t = t ^ (t >> 15)
    t = _mul32(t, 0x846CA68B)
    t = t ^ (t >> 16)
    return t


def stream_key(*parts: int) -> int:
    """Fold integers into one 32-bit stream key."""
    h = 0x6A09E667
    for p in parts:
        h = mix32_int(h ^ mix32_int(int(p) & MASK32))
        h = mix32_int(h + 0x9E3779B9)
    return h


def hash_stream(idx: torch.Tensor, key) -> torch.Tensor:
    """32-bit draws for counters ``idx`` (int64, < 2^32) of stream ``key``.

    ``key`` is an int or an int64 tensor broadcastable against ``idx``.
    """
    if isinstance(key, int):
        k2 = mix32_int(key ^ 0x5BD1E995)
    else:
        k2 = mix32(key ^ 0x5BD1E995)
    return mix32((mix32(idx ^ key) + k2) & MASK32)


# ---------------------------------------------------------------------------
# distributions
# ---------------------------------------------------------------------------
def _f32_to_bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


_TABLE_BITS: Optional[np.ndarray] = None
_TABLES: Dict[str, torch.Tensor] = {}


def normal_table_bits() -> np.ndarray:
    """bf16 bit patterns of the 65536 N(0,1) quantiles at (u + 0.5) / 65536."""
    global _TABLE_BITS
    if _TABLE_BITS is None:
        nd = statistics.NormalDist()
        vals = np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)], dtype=np.float64)
        _TABLE_BITS = _f32_to_bf16_bits_rne(vals.astype(np.float32))
    return _TABLE_BITS


def _normal_table(device) -> torch.Tensor:
    key = str(torch.device(device))
    if key not in _TABLES:
        bits = normal_table_bits().astype(np.uint32) << np.uint32(16)
        _TABLES[key] = torch.from_numpy(bits.view(np.float32).copy()).to(device)
    return _TABLES[key]


def normal_from_hash(h: torch.Tensor) -> torch.Tensor:
    """fp32 tensor of bf16-exact N(0,1) values."""
    return _normal_table(h.device)[h & 0xFFFF]


def uniform_from_hash(h: torch.Tensor) -> torch.Tensor:
    """fp32 U[0,1) on a 2^-24 grid (exact in fp32)."""
    return (h >> 8).to(torch.float32) * (1.0 / 16777216.0)


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


# ---------------------------------------------------------------------------
# workload pieces
# ---------------------------------------------------------------------------
def seq_lens(w: Workload, seed: int) -> List[int]:
    lo, hi = w.ctx
    if lo == hi:
        return [lo] * w.batch
    steps = (hi - lo) // 32 + 1
    return [lo + 32 * (mix32_int(stream_key(seed, _LEN, b)) % steps) for b in range(w.batch)]


def _attempts(w: Workload, attempts) -> np.ndarray:
    if attempts is None:
        return np.zeros((w.batch, w.n_kv_heads), dtype=np.int64)
    a = np.asarray(attempts, dtype=np.int64)
    assert a.shape == (w.batch, w.n_kv_heads)
    return a


def gen_group_query(w: Workload, seed: int, layer: int, b: int, g: int, attempt: int = 0):
    """(q, q_spec) of one (request, KV head) group as bf16 ``[r][d]`` (q_spec may be None)."""
    r, d = w.group_size, w.head_dim
    idx = torch.arange(r * d, dtype=torch.int64)
    n = normal_from_hash(hash_stream(idx, stream_key(seed, _Q, layer, b, g, attempt)))
    q = _bf16(n).view(r, d)
    if w.spec_sigma is None:
        return q, None
    e = normal_from_hash(hash_stream(idx, stream_key(seed, _QS, layer, b, g, attempt)))
    sig = torch.tensor(w.spec_sigma, dtype=torch.float32)
    return q, _bf16(n + sig * e).view(r, d)


def gen_group_query_step(w: Workload, seed: int, layer: int, b: int, g: int, step: int, drift: float,
                         attempt: int = 0):
    """(q, q_spec) of one group at decode step ``step`` (bf16 ``[r][d]``; q_spec may be None).

    q = bf16(n + drift * e_step), q_spec = bf16(n + drift * e_{step+1} + sigma * f_step):
    the speculative query is a noisy estimate of the next step's query.
    """
    r, d = w.group_size, w.head_dim
    idx = torch.arange(r * d, dtype=torch.int64)
    n = normal_from_hash(hash_stream(idx, stream_key(seed, _Q, layer, b, g, attempt)))
    dr = torch.tensor(drift, dtype=torch.float32)

    def e(s):
        return normal_from_hash(hash_stream(idx, stream_key(seed, _QD, layer, b, g, attempt, s)))
    x = n if drift == 0 else n + dr * e(step)
    q = _bf16(x).view(r, d)
    if w.spec_sigma is None:
        return q, None
    key = (seed, _QS, layer, b, g, attempt) + ((step,) if step else ())
    f = normal_from_hash(hash_stream(idx, stream_key(*key)))
    y = n if drift == 0 else n + dr * e(step + 1)
    sig = torch.tensor(w.spec_sigma, dtype=torch.float32)
    return q, _bf16(y + sig * f).view(r, d)


def gen_queries_step(w: Workload, seed: int, layer: int, step: int, drift: float, attempts=None):
    """(q, q_spec) bf16 CPU tensors ``[b][Hq][d]`` of decode step ``step``."""
    a = _attempts(w, attempts)
    r, d = w.group_size, w.head_dim
    q = torch.empty(w.batch, w.n_q_heads, d, dtype=torch.bfloat16)
    qs = None if w.spec_sigma is None else torch.empty_like(q)
    for b in range(w.batch):
        for g in range(w.n_kv_heads):
            qg, qsg = gen_group_query_step(w, seed, layer, b, g, step, drift, int(a[b, g]))
            q[b, g * r:(g + 1) * r] = qg
            if qs is not None:
                qs[b, g * r:(g + 1) * r] = qsg
    return q, qs


def gen_queries(w: Workload, seed: int, layer: int, attempts=None):
    """(q, q_spec) bf16 CPU tensors ``[b][Hq][d]``; q_spec is None without speculation."""
    a = _attempts(w, attempts)
    r, d = w.group_size, w.head_dim
    q = torch.empty(w.batch, w.n_q_heads, d, dtype=torch.bfloat16)
    qs = None if w.spec_sigma is None else torch.empty_like(q)
    for b in range(w.batch):
        for g in range(w.n_kv_heads):
            qg, qsg = gen_group_query(w, seed, layer, b, g, int(a[b, g]))
            q[b, g * r:(g + 1) * r] = qg
            if qs is not None:
                qs[b, g * r:(g + 1) * r] = qsg
    return q, qs


def _plant_direction(w: Workload, q_group: torch.Tensor) -> torch.Tensor:
    """fp32 ``[d]`` = beta * (sum_h q_h) / |sum_h q_h| (host fp64, one rounding to fp32)."""
    u = q_group.to(torch.float64).sum(dim=0)
    u = u / torch.linalg.vector_norm(u)
    return (w.plant_beta * u).to(torch.float32)


def planted_blocks(w: Workload, seed: int, layer: int, b: int, g: int, n_cand: int) -> torch.Tensor:
    """Ascending ids of the planted blocks / tokens of group (b, g) among n_cand candidates."""
    key = stream_key(seed, _PLANT, layer, b, g)
    if w.plant == "blocks":
        ids = torch.arange(n_cand, dtype=torch.int64)
        order = torch.argsort(hash_stream(ids, key) * 2**20 + ids)
        return torch.sort(order[: w.n_planted]).values
    if w.plant == "token_runs":
        n = w.n_planted
        n_iso = int(round(0.6 * n))
        remaining = n - n_iso
        seg_len = [1] * n_iso
        i = 0
        while remaining > 0:
            L = 2 + mix32_int(stream_key(key, _SEG, i)) % 63
            L = min(L, remaining)
            if remaining - L == 1:
                L = remaining
            seg_len.append(L)
            remaining -= L
            i += 1
        ns = len(seg_len)
        seg_ids = torch.arange(ns, dtype=torch.int64)
        perm = torch.argsort(hash_stream(seg_ids, stream_key(key, 1)) * 2**20 + seg_ids)
        lens = torch.tensor(seg_len, dtype=torch.int64)[perm]
        span = n_cand - (n - ns) - (ns - 1)           # positions after compressing segments + gaps
        pos_ids = torch.arange(span, dtype=torch.int64)
        pos = torch.sort(torch.argsort(hash_stream(pos_ids, stream_key(key, 2)) * 2**20 + pos_ids)[:ns]).values
        # start_i = pos_i + sum_{j<i}(L_j - 1) + i = pos_i + sum_{j<i} L_j: distinct
        # sorted pos keep one unplanted token between consecutive segments, and the
        # last segment ends by pos_max + n - 1 <= n_cand - 1.
        starts = pos + (torch.cumsum(lens, 0) - lens)
        out = torch.cat([torch.arange(s, s + L) for s, L in zip(starts.tolist(), lens.tolist())])
        return torch.sort(out).values
    raise ValueError(w.plant)


def gen_lowrank_factors(w: Workload, seed: int, layer: int, b: int, n_tok: int, device="cpu"):
    """Rank-R key factors of request b: coefficients bf16 ``[Hkv][n_tok][R]``, basis bf16 ``[Hkv][R][d]``."""
    H, d, R = w.n_kv_heads, w.head_dim, w.lowrank_rank
    cidx = torch.arange(n_tok * R, dtype=torch.int64, device=device).view(1, -1)
    kc = torch.tensor([stream_key(seed, _LRC, layer, b, g) for g in range(H)], dtype=torch.int64,
                      device=device).view(H, 1)
    coef = _bf16(normal_from_hash(hash_stream(cidx, kc))).view(H, n_tok, R)
    bidx = torch.arange(R * d, dtype=torch.int64, device=device).view(1, -1)
    kb = torch.tensor([stream_key(seed, _LRB, layer, b, g) for g in range(H)], dtype=torch.int64,
                      device=device).view(H, 1)
    scale = torch.tensor(1.0 / math.sqrt(R), dtype=torch.float32)
    basis = _bf16(normal_from_hash(hash_stream(bidx, kb)) * scale.to(device)).view(H, R, d)
    return coef, basis


def lowrank_product(coef: torch.Tensor, basis: torch.Tensor) -> torch.Tensor:
    """bf16 ``[H][n][d]`` = sum over j ascending of fp32(coef[..., j]) * fp32(basis[j]),
    each product and each partial sum rounded to fp32 (separate multiply and add)."""
    H, n, R = coef.shape
    acc = torch.zeros(H, n, basis.shape[2], dtype=torch.float32, device=coef.device)
    for j in range(R):
        prod = coef[:, :, j:j + 1].to(torch.float32) * basis[:, j:j + 1, :].to(torch.float32)
        acc = acc + prod
    return _bf16(acc)


def gen_request_kv(w: Workload, seed: int, layer: int, b: int, n_tok: int, q_req: torch.Tensor,
                   device="cpu"):
    """K, V of request b as bf16 ``[Hkv][n_tok][d]`` on ``device``.

    ``q_req`` (``[Hq][d]`` bf16, CPU) is only used for the planting direction.
    """
    H, d = w.n_kv_heads, w.head_dim
    idx = torch.arange(n_tok * d, dtype=torch.int64, device=device).view(1, -1)
    kk = torch.tensor([stream_key(seed, _K, layer, b, g) for g in range(H)], dtype=torch.int64,
                      device=device).view(H, 1)
    kv = torch.tensor([stream_key(seed, _V, layer, b, g) for g in range(H)], dtype=torch.int64,
                      device=device).view(H, 1)
    V = _bf16(normal_from_hash(hash_stream(idx, kv))).view(H, n_tok, d)
    n = normal_from_hash(hash_stream(idx, kk)).view(H, n_tok, d)
    if w.key_dist == "normal":
        K = n
    elif w.key_dist == "channel_scaled":
        cidx = torch.arange(d, dtype=torch.int64, device=device).view(1, -1)
        ks = torch.tensor([stream_key(seed, _KS, layer, g) for g in range(H)], dtype=torch.int64,
                          device=device).view(H, 1)
        s = 0.5 + 1.5 * uniform_from_hash(hash_stream(cidx, ks))      # [H][d]
        K = n * s.view(H, 1, d)
    elif w.key_dist == "clustered":
        m_idx = torch.arange(w.n_centroids * d, dtype=torch.int64, device=device).view(1, -1)
        km = torch.tensor([stream_key(seed, _MU, layer, b, g) for g in range(H)], dtype=torch.int64,
                          device=device).view(H, 1)
        mu = normal_from_hash(hash_stream(m_idx, km)).view(H, w.n_centroids, d)
        n_blk = (n_tok + w.block_size - 1) // w.block_size
        j_idx = torch.arange(n_blk, dtype=torch.int64, device=device).view(1, -1)
        ka = torch.tensor([stream_key(seed, _ASSIGN, layer, b, g) for g in range(H)],
                          dtype=torch.int64, device=device).view(H, 1)
        assign = hash_stream(j_idx, ka) % w.n_centroids                 # [H][n_blk]
        tok_assign = assign.repeat_interleave(w.block_size, dim=1)[:, :n_tok]
        mu_tok = torch.gather(mu, 1, tok_assign.unsqueeze(-1).expand(H, n_tok, d))
        K = mu_tok + torch.tensor(w.centroid_sigma, dtype=torch.float32, device=device) * n
    elif w.key_dist == "lowrank":
        K = lowrank_product(*gen_lowrank_factors(w, seed, layer, b, n_tok, device=device))
    else:
        raise ValueError(w.key_dist)
    K = _bf16(K)
    if w.plant is not None:
        r = w.group_size
        n_cand = (n_tok - w.window) // w.block_size
        for g in range(H):
            ids = planted_blocks(w, seed, layer, b, g, n_cand)
            if w.block_size > 1:
                toks = (ids.view(-1, 1) * w.block_size + torch.arange(w.block_size)).view(-1)
            else:
                toks = ids
            toks = toks.to(device)
            shift = _plant_direction(w, q_req[g * r:(g + 1) * r]).to(device)
            K[g, toks] = _bf16(K[g, toks].to(torch.float32) + shift.view(1, d))
    return K, V


class LayerInputs:
    """Packed host K/V ``[b][Hkv][len_b][d]`` (bf16) of one layer plus its queries."""

    def __init__(self, k, v, q, q_spec, lens):
        self.k, self.v, self.q, self.q_spec, self.lens = k, v, q, q_spec, lens


def layer_numel(w: Workload, lens: List[int]) -> int:
    return sum(lens) * w.n_kv_heads * w.head_dim


def fill_lowrank(w: Workload, seed: int, layer: int, coef_out: torch.Tensor, basis_out: torch.Tensor,
                 lens: List[int], device="cpu") -> None:
    """One layer's low-rank key factors, packed like the host K: coefficients
    ``[b][Hkv][len_b][R]`` into flat ``coef_out``, basis ``[b][Hkv][R][d]`` into ``basis_out``."""
    off = 0
    H, d, R = w.n_kv_heads, w.head_dim, w.lowrank_rank
    for b, n_tok in enumerate(lens):
        coef, basis = gen_lowrank_factors(w, seed, layer, b, n_tok, device=device)
        coef_out[off:off + coef.numel()].copy_(coef.reshape(-1))
        basis_out[b * H * R * d:(b + 1) * H * R * d].copy_(basis.reshape(-1))
        off += coef.numel()


def fill_layer(w: Workload, seed: int, layer: int, k_out: torch.Tensor, v_out: torch.Tensor,
               q: torch.Tensor, lens: List[int], device="cpu") -> None:
    """Write one layer's packed K/V into flat bf16 tensors (host or device).

    Values are generated on ``device`` and copied into ``k_out``/``v_out``.
    """
    off = 0
    for b, n_tok in enumerate(lens):
        K, V = gen_request_kv(w, seed, layer, b, n_tok, q[b], device=device)
        n = K.numel()
        k_out[off:off + n].copy_(K.reshape(-1))
        v_out[off:off + n].copy_(V.reshape(-1))
        off += n


def make_layer(w: Workload, seed: int, layer: int = 0, attempts=None, device="cpu",
               pin: bool = False) -> LayerInputs:
    """Convenience for small workloads: one layer's inputs as flat CPU tensors."""
    lens = seq_lens(w, seed)
    q, qs = gen_queries(w, seed, layer, attempts)
    n = layer_numel(w, lens)
    k = torch.empty(n, dtype=torch.bfloat16, pin_memory=pin)
    v = torch.empty(n, dtype=torch.bfloat16, pin_memory=pin)
    fill_layer(w, seed, layer, k, v, q, lens, device=device)
    return LayerInputs(k, v, q, qs, lens)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a bf16 CPU tensor's bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
