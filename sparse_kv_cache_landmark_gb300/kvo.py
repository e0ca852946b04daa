"""Python binding of libkvo (the C ABI in include/kvo.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; this module
turns torch tensors into pointers, allocates outputs with torch, and raises
``KvoError`` on any non-OK status.  There is no fallback: without the built
library or a CUDA device every call fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvo.so")

KVO_OK, KVO_ERR_INVALID, KVO_ERR_CUDA, KVO_ERR_OOM, KVO_ERR_TIMEOUT, KVO_ERR_STATE, KVO_ERR_DEVICE = range(7)
DEV_BAD_BLOCK_ID, DEV_BAD_SLOT, DEV_BAD_COUNT, DEV_UNSORTED, DEV_TIMEOUT = 1, 2, 4, 8, 16

EXPORTS = ["kv_offload_init", "kv_offload_destroy", "select_topk", "index_diff", "gather_coalesced",
           "sparse_decode_attn", "merge_lse", "kvo_decode_step", "kvo_reset_prediction", "kvo_get_stream",
           "kvo_device_status", "kvo_landmarks", "kvo_buffer", "kvo_info", "kvo_profile", "kvo_profile_read",
           "kvo_last_error", "sparse_decode_attn_static", "kvo_set_gather_shape", "kvo_set_gather_engine", "kvo_profile_trace", "sparse_decode_attn_cobatch",
           "kvo_decode_step_dual", "kvo_set_gather_reserve", "kvo_set_graphs", "kvo_append",
           "kvo_set_attn_impl", "kvo_set_select_impl", "kvo_resident_slots", "kvo_resident_fetched",
           "kvo_set_prefetch_budget", "kvo_set_lowrank_keys", "kvo_plan_attention", "kvo_plan_select", "kvo_set_wait_test",
           "kvo_set_spec_policy", "kvo_spec_stats"]
PROFILE_KINDS = ["select", "diff", "coalesce", "gather_prefetch", "gather_urgent", "attention", "recon"]


class KvoError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kvo status {status}: {msg}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("window", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("seq_lens", ctypes.POINTER(ctypes.c_int32)), ("max_append", ctypes.c_int32),
                ("resident", ctypes.c_int32)]


_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libkvo.so (built by ``build.py``); raises if it is missing."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvo.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, VP = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        L.kv_offload_init.argtypes = [ctypes.POINTER(_Config), P, P, P, P, ctypes.POINTER(P)]
        L.kv_offload_destroy.argtypes = [P]
        L.select_topk.argtypes = [P, I, VP, VP, VP, VP, VP]
        L.index_diff.argtypes = [P, VP, VP, VP, VP, VP, VP]
        L.gather_coalesced.argtypes = [P, I, I, VP, VP, I, I, VP, VP, VP]
        L.sparse_decode_attn.argtypes = [P, I, I, VP, VP, VP, VP, I, VP]
        L.merge_lse.argtypes = [VP, VP, VP, VP, VP, VP, I, I, VP]
        L.kvo_decode_step.argtypes = [P, VP, VP, VP, VP, VP]
        L.kvo_decode_step_dual.argtypes = [P, VP, VP, VP, VP, VP, VP, VP]
        L.sparse_decode_attn_cobatch.argtypes = [P, I, I, VP, VP, VP, VP, VP, VP, VP, I, VP]
        L.kvo_reset_prediction.argtypes = [P]
        L.kvo_get_stream.argtypes = [P, I, ctypes.POINTER(P)]
        L.kvo_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32), VP]
        L.kvo_landmarks.argtypes = [P, I, VP, VP]
        L.kvo_buffer.argtypes = [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]
        L.kvo_info.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
        L.kvo_profile.argtypes = [P, I]
        L.kvo_profile_read.argtypes = [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), I]
        L.sparse_decode_attn_static.argtypes = [VP, VP, VP, VP, VP, VP, VP, VP, VP] + [I] * 8 + [VP]
        L.kvo_set_gather_shape.argtypes = [P, I, I, I]
        L.kvo_set_gather_engine.argtypes = [P, I, I]
        L.kvo_set_gather_reserve.argtypes = [P, I]
        L.kvo_set_graphs.argtypes = [P, I]
        L.kvo_set_attn_impl.argtypes = [P, I, I]
        L.kvo_set_select_impl.argtypes = [P, I]
        L.kvo_resident_slots.argtypes = [P, I, ctypes.POINTER(ctypes.c_int32)]
        L.kvo_resident_fetched.argtypes = [P, ctypes.POINTER(ctypes.c_int64), I]
        L.kvo_set_prefetch_budget.argtypes = [P, I]
        L.kvo_set_lowrank_keys.argtypes = [P, I, I, VP, VP]
        L.kvo_append.argtypes = [P, VP, VP, VP]
        L.kvo_set_wait_test.argtypes = [P, ctypes.c_int64, I]
        L.kvo_set_spec_policy.argtypes = [P, I]
        L.kvo_spec_stats.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
        DP, IP = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32)
        L.kvo_profile_trace.argtypes = [P, DP, DP, IP, IP, I, ctypes.POINTER(ctypes.c_int)]
        L.kvo_last_error.argtypes = [P]
        L.kvo_last_error.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "kvo_last_error":
                getattr(L, name).restype = ctypes.c_int
        _LIB = L
    return _LIB


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


CUDA_STREAM_LEGACY = 0x1   # cudaStreamLegacy: the legacy default stream


def _stream(stream) -> ctypes.c_void_p:
    """Handle of ``stream`` (default: torch's current stream) for the C ABI.

    The ABI reads NULL as "the context's own compute stream", so torch's
    default stream (handle 0) is passed as cudaStreamLegacy instead.
    """
    if stream is None:
        stream = torch.cuda.current_stream()
    h = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(h or CUDA_STREAM_LEGACY)


def _check(st: int, ctx=None):
    if st != KVO_OK:
        msg = lib().kvo_last_error(ctx)
        raise KvoError(st, msg.decode() if msg else "")


def merge_lse(o1, lse1, o2, lse2, o=None, lse=None, stream=None):
    """Fuse two attention parts by log-sum-exp (C: merge_lse). fp32 CUDA tensors [rows][d], [rows]."""
    rows, d = o1.shape
    o = torch.empty_like(o1) if o is None else o
    lse = torch.empty_like(lse1) if lse is None else lse
    _check(lib().merge_lse(_ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), _ptr(o), _ptr(lse), rows, d, _stream(stream)))
    return o, lse


def plan_select(blocks_per_group, n_sms: int, impl: int = 1) -> dict:
    """Launch plan of the selection kernels (C: kvo_plan_select; host only):
    rows per thread, the most CTAs a group needs, the ticket kernel's CTAs, and
    the cluster kernel's CTAs per cluster (0: the ticket kernel runs)."""
    blocks = (ctypes.c_int32 * len(blocks_per_group))(*[int(x) for x in blocks_per_group])
    out = (ctypes.c_int32 * 4)()
    _check(lib().kvo_plan_select(len(blocks_per_group), blocks, n_sms, impl, out))
    return {"rows_per_thread": out[0], "ctas_per_group": out[1], "ctas": out[2], "cluster_ctas": out[3]}


def plan_attention(n_groups: int, sparse_tokens: int, window_tokens: int, grid: int):
    """Work split of the TMA-staged attention (C: kvo_plan_attention; host only).

    Returns (items int32 [n][4] = {group, part, first tile, tiles}, cta int32
    [grid_used + 1] = first item of each CTA's range, then the item count).
    """
    n = ctypes.c_int32(0)
    g = ctypes.c_int32(0)
    L = lib()
    _check(L.kvo_plan_attention(n_groups, sparse_tokens, window_tokens, grid, None, 0, None, ctypes.byref(n),
                                ctypes.byref(g)))
    items = torch.empty(max(1, n.value), 4, dtype=torch.int32)
    cta = torch.empty(g.value + 1, dtype=torch.int32)
    _check(L.kvo_plan_attention(n_groups, sparse_tokens, window_tokens, grid,
                                ctypes.c_void_p(items.data_ptr()), items.shape[0],
                                ctypes.c_void_p(cta.data_ptr()), ctypes.byref(n), ctypes.byref(g)))
    return items[:n.value], cta


def sparse_decode_attn_static(q, k_buf, v_buf, slot_of_true, k_win, v_win, *, batch, n_q_heads, n_kv_heads,
                              head_dim, block_size, top_k, window, fuse_window_merge=True, o=None, lse=None,
                              status=None, stream=None):
    """Context-free attention that allocates no device memory in the library (C: sparse_decode_attn_static).

    Meant for callers that cannot call cudaMalloc: code whose device memory all
    belongs to another allocator (a framework arena or a pool sized at start-up)
    and decode loops that cannot afford the implicit synchronisation of
    cudaMalloc / cudaFree.  The library's scratch is a fixed 24 MiB static device
    array shared by every call, so calls must not overlap on the GPU.
    ``k_buf``/``v_buf`` are bf16 CUDA tensors laid out like a ping-pong half,
    [G][2k][B][d].  Pass ``o``/``lse`` (and ``status``) to keep this wrapper from
    allocating its outputs with torch (it allocates them on ``q``'s device).
    Every buffer's dtype, contiguity, size and device is checked against the
    shape arguments before the call; a mismatch raises ``KvoError``.  A slot
    outside [0, 2k) is reported in ``status`` (int32, optional); without a
    status word such errors are dropped.
    """
    rows = batch * n_q_heads
    parts = 1 if fuse_window_merge else 2
    G = batch * n_kv_heads
    # this call has no context to size the buffers by: a short buffer would be
    # an out-of-bounds device access, so every buffer is checked here first
    need = [("q", q, torch.bfloat16, rows * head_dim),
            ("k_buf", k_buf, torch.bfloat16, G * 2 * top_k * block_size * head_dim),
            ("v_buf", v_buf, torch.bfloat16, G * 2 * top_k * block_size * head_dim),
            ("slot_of_true", slot_of_true, torch.int32, G * top_k)]
    if window > 0:
        need += [("k_win", k_win, torch.bfloat16, G * window * head_dim),
                 ("v_win", v_win, torch.bfloat16, G * window * head_dim)]
    if o is not None:
        need.append(("o", o, torch.float32, parts * rows * head_dim))
    if lse is not None:
        need.append(("lse", lse, torch.float32, parts * rows))
    if status is not None:
        need.append(("status", status, torch.int32, 1))
    for name, t, dt, n in need:
        if t is None:
            raise KvoError(KVO_ERR_INVALID, f"{name} is required")
        if t.dtype != dt:
            raise KvoError(KVO_ERR_INVALID, f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise KvoError(KVO_ERR_INVALID, f"{name} must be contiguous")
        if t.numel() < n:
            raise KvoError(KVO_ERR_INVALID, f"{name} holds {t.numel()} elements, the shape needs {n}")
    devs = {t.device for _, t, _, _ in need}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise KvoError(KVO_ERR_INVALID, f"all buffers must be on one CUDA device, got {sorted(map(str, devs))}")
    if o is None:
        o = torch.empty(parts, rows, head_dim, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(parts, rows, dtype=torch.float32, device=q.device)
    _check(lib().sparse_decode_attn_static(_ptr(q), _ptr(k_buf), _ptr(v_buf), _ptr(slot_of_true), _ptr(k_win),
                                           _ptr(v_win), _ptr(o), _ptr(lse), _ptr(status), batch, n_q_heads,
                                           n_kv_heads, head_dim, block_size, top_k, window,
                                           int(bool(fuse_window_merge)), _stream(stream)))
    return o, lse


class Context:
    """A KV cache in pinned host memory plus the library's device state (C: kv_offload_init).

    ``k_host[l]``/``v_host[l]``: pinned CPU bf16 tensors, packed [b][Hkv][len_b][d];
    ``k_win[l]``/``v_win[l]``: CUDA bf16 tensors [b][Hkv][W][d] (None when W == 0).
    The tensors must outlive the context; the context keeps references to them.
    """

    def __init__(self, *, batch, n_q_heads, n_kv_heads, head_dim, block_size, top_k, window, n_layers,
                 seq_lens: Sequence[int], k_host: List[torch.Tensor], v_host: List[torch.Tensor],
                 k_win: Optional[List[torch.Tensor]] = None, v_win: Optional[List[torch.Tensor]] = None,
                 max_append: int = 0, resident: bool = False):
        L = lib()
        self._lens = (ctypes.c_int32 * batch)(*[int(x) for x in seq_lens])
        self.cfg = _Config(batch, n_q_heads, n_kv_heads, head_dim, block_size, top_k, window, n_layers, self._lens,
                           max_append, int(bool(resident)))
        self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim = batch, n_q_heads, n_kv_heads, head_dim
        self.block_size, self.top_k, self.window, self.n_layers = block_size, top_k, window, n_layers
        self.G = batch * n_kv_heads
        self._keep = (list(k_host), list(v_host), list(k_win or []), list(v_win or []))
        arr = lambda ts: (ctypes.c_void_p * n_layers)(*[t.data_ptr() for t in ts]) if ts else None
        self._kh, self._vh = arr(k_host), arr(v_host)
        self._kw, self._vw = arr(k_win), arr(v_win)
        out = ctypes.c_void_p()
        _check(L.kv_offload_init(ctypes.byref(self.cfg), self._kh, self._vh, self._kw, self._vw, ctypes.byref(out)))
        self.ctx = out

    def close(self):
        if getattr(self, "ctx", None):
            lib().kv_offload_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _c(self, st):
        _check(st, self.ctx)

    def _i32(self, *shape):
        return torch.empty(*shape, dtype=torch.int32, device="cuda")

    def select_topk(self, layer, q, q_spec=None, idx_true=None, idx_pred=None, stream=None):
        idx_true = self._i32(self.G, self.top_k) if idx_true is None else idx_true
        if q_spec is not None and idx_pred is None:
            idx_pred = self._i32(self.G, self.top_k)
        self._c(lib().select_topk(self.ctx, layer, _ptr(q), _ptr(q_spec), _ptr(idx_true),
                                  _ptr(idx_pred) if q_spec is not None else None, _stream(stream)))
        return idx_true, (idx_pred if q_spec is not None else None)

    def index_diff(self, idx_true, idx_pred=None, stream=None):
        miss = self._i32(self.G, self.top_k)
        cnt = self._i32(self.G)
        slot = self._i32(self.G, self.top_k)
        self._c(lib().index_diff(self.ctx, _ptr(idx_true), _ptr(idx_pred), _ptr(miss), _ptr(cnt), _ptr(slot),
                                 _stream(stream)))
        return miss, cnt, slot

    def gather_coalesced(self, layer, buf, idx, cnt=None, slot_base=0, urgent=False, want_runs=True, stream=None):
        runs = self._i32(self.G, self.top_k, 4) if want_runs else None
        nruns = self._i32(self.G) if want_runs else None
        self._c(lib().gather_coalesced(self.ctx, layer, buf, _ptr(idx), _ptr(cnt), slot_base, int(bool(urgent)),
                                       _ptr(runs), _ptr(nruns), _stream(stream)))
        return runs, nruns

    def sparse_decode_attn(self, layer, buf, q, slot_of_true, fuse_window_merge=True, o=None, lse=None, stream=None):
        rows = self.batch * self.n_q_heads
        parts = 1 if fuse_window_merge else 2
        if o is None:
            o = torch.empty(parts, rows, self.head_dim, dtype=torch.float32, device="cuda")
        if lse is None:
            lse = torch.empty(parts, rows, dtype=torch.float32, device="cuda")
        self._c(lib().sparse_decode_attn(self.ctx, layer, buf, _ptr(q), _ptr(slot_of_true), _ptr(o), _ptr(lse),
                                         int(bool(fuse_window_merge)), _stream(stream)))
        return o, lse

    def sparse_decode_attn_cobatch(self, layer, buf, q, q_spec, slot_of_true, fuse_window_merge=True, stream=None):
        """Co-batched attention of q and q_spec over the same blocks (C: sparse_decode_attn_cobatch)."""
        rows = self.batch * self.n_q_heads
        parts = 1 if fuse_window_merge else 2
        mk = lambda *sh: torch.empty(*sh, dtype=torch.float32, device="cuda")
        o, lse, os_, ls_ = mk(parts, rows, self.head_dim), mk(parts, rows), mk(parts, rows, self.head_dim), mk(parts, rows)
        self._c(lib().sparse_decode_attn_cobatch(self.ctx, layer, buf, _ptr(q), _ptr(q_spec), _ptr(slot_of_true),
                                                 _ptr(o), _ptr(lse), _ptr(os_), _ptr(ls_),
                                                 int(bool(fuse_window_merge)), _stream(stream)))
        return o, lse, os_, ls_

    def decode_step_dual(self, q, q_spec, stream=None):
        """Pipelined step with co-batched attention (C: kvo_decode_step_dual) -> (o, lse, o_spec, lse_spec)."""
        rows = self.batch * self.n_q_heads
        mk = lambda *sh: torch.empty(*sh, dtype=torch.float32, device="cuda")
        o, lse = mk(self.n_layers, rows, self.head_dim), mk(self.n_layers, rows)
        os_, ls_ = mk(self.n_layers, rows, self.head_dim), mk(self.n_layers, rows)
        self._c(lib().kvo_decode_step_dual(self.ctx, _ptr(q), _ptr(q_spec), _ptr(o), _ptr(lse), _ptr(os_),
                                           _ptr(ls_), _stream(stream)))
        return o, lse, os_, ls_

    def decode_step(self, q, q_spec=None, o=None, lse=None, stream=None):
        """One pipelined decode step over every layer (C: kvo_decode_step)."""
        rows = self.batch * self.n_q_heads
        if o is None:
            o = torch.empty(self.n_layers, rows, self.head_dim, dtype=torch.float32, device="cuda")
        if lse is None:
            lse = torch.empty(self.n_layers, rows, dtype=torch.float32, device="cuda")
        self._c(lib().kvo_decode_step(self.ctx, _ptr(q), _ptr(q_spec), _ptr(o), _ptr(lse), _stream(stream)))
        return o, lse

    def append(self, k_new, v_new, stream=None):
        """Grow every request by one token (C: kvo_append); k_new, v_new: CUDA bf16 [L][b][Hkv][d]."""
        self._c(lib().kvo_append(self.ctx, _ptr(k_new), _ptr(v_new), _stream(stream)))

    def reset_prediction(self):
        self._c(lib().kvo_reset_prediction(self.ctx))

    def get_stream(self, which: int) -> int:
        out = ctypes.c_void_p()
        self._c(lib().kvo_get_stream(self.ctx, which, ctypes.byref(out)))
        return out.value or 0

    def device_status(self, stream=None) -> int:
        code = ctypes.c_int32(0)
        st = lib().kvo_device_status(self.ctx, ctypes.byref(code), _stream(stream))
        if st not in (KVO_OK, KVO_ERR_DEVICE):
            self._c(st)
        return int(code.value)

    def info(self):
        out = (ctypes.c_int64 * 4)()
        self._c(lib().kvo_info(self.ctx, out))
        return {"C_max": out[0], "landmark_bytes": out[1], "pingpong_bytes": out[2], "scratch_bytes": out[3]}

    def set_gather_shape(self, ctas: int = 0, threads: int = 256, unroll: int = 4):
        self._c(lib().kvo_set_gather_shape(self.ctx, ctas, threads, unroll))

    def set_gather_engine(self, engine: int, drivers: int = 0):
        """0: lane-load gather, 1: TMA bulk-copy gather with ``drivers`` driver warps."""
        self._c(lib().kvo_set_gather_engine(self.ctx, engine, drivers))

    def set_graphs(self, enable: bool):
        """Replay warm decode steps from captured CUDA graphs (C: kvo_set_graphs)."""
        self._c(lib().kvo_set_graphs(self.ctx, int(bool(enable))))

    def resident_slots(self, layer: int) -> torch.Tensor:
        """Slot table of layer ``layer``'s resident set, int32 ``[G][2k]`` (-1 empty) (C: kvo_resident_slots)."""
        out = torch.empty(self.G, 2 * self.top_k, dtype=torch.int32)
        self._c(lib().kvo_resident_slots(self.ctx, layer,
                                         ctypes.cast(out.data_ptr(), ctypes.POINTER(ctypes.c_int32))))
        return out

    def set_lowrank_keys(self, layer: int, rank: int, coef: Optional[torch.Tensor], basis: Optional[torch.Tensor]):
        """Rebuild layer ``layer``'s missed keys from rank-``rank`` factors (C: kvo_set_lowrank_keys).

        coef: CUDA bf16 packed like the host K with ``rank`` values per token; basis: CUDA bf16
        ``[b][Hkv][rank][d]``.  The tensors must outlive their use; the context keeps references.
        """
        self._lr = getattr(self, "_lr", {})
        self._lr[layer] = (coef, basis)
        self._c(lib().kvo_set_lowrank_keys(self.ctx, layer, rank, _ptr(coef), _ptr(basis)))

    def set_prefetch_budget(self, blocks: int):
        """Cap prefetch fetches per group, layer and step (-1: no cap) (C: kvo_set_prefetch_budget)."""
        self._c(lib().kvo_set_prefetch_budget(self.ctx, blocks))

    def set_spec_policy(self, mode: int):
        """0: prefetch every layer's prediction; 1: per layer, only while it pays (C: kvo_set_spec_policy)."""
        self._c(lib().kvo_set_spec_policy(self.ctx, int(mode)))

    def spec_stats(self):
        """Per layer (blocks prefetched, prefetched blocks used, prefetch on) (C: kvo_spec_stats)."""
        out = (ctypes.c_int64 * (3 * self.n_layers))()
        self._c(lib().kvo_spec_stats(self.ctx, out))
        return [(int(out[3 * l]), int(out[3 * l + 1]), int(out[3 * l + 2])) for l in range(self.n_layers)]

    def resident_fetched(self, reset: bool = False):
        """(urgent, prefetch) blocks fetched since init or the last reset (C: kvo_resident_fetched)."""
        out = (ctypes.c_int64 * 2)()
        self._c(lib().kvo_resident_fetched(self.ctx, out, int(bool(reset))))
        return int(out[0]), int(out[1])

    def set_attn_impl(self, impl: int, ctas: int = 0):
        """Attention kernel: 0 register-direct loads, 1 TMA-staged persistent with
        ``ctas`` CTAs (0: as many as fit), 2 (default) group-split clusters of
        ``ctas`` CTAs per group (0: automatic) (C: kvo_set_attn_impl)."""
        self._c(lib().kvo_set_attn_impl(self.ctx, impl, ctas))

    def set_select_impl(self, impl: int):
        """Selection kernel: 0 ticket, 2 one cluster per group where a group's
        CTAs fit one, 1 (default) the cluster kernel where the ticket kernel's
        tail would be long and exposed (C: kvo_set_select_impl)."""
        self._c(lib().kvo_set_select_impl(self.ctx, impl))

    def set_wait_test(self, limit_ns: int = 2_000_000_000, skip_tile: int = -1):
        """Bounded-wait test switch of the TMA-staged attention (C: kvo_set_wait_test)."""
        self._c(lib().kvo_set_wait_test(self.ctx, int(limit_ns), int(skip_tile)))

    def set_gather_reserve(self, smem_bytes: int):
        self._c(lib().kvo_set_gather_reserve(self.ctx, smem_bytes))

    def profile(self, enable: bool):
        self._c(lib().kvo_profile(self.ctx, int(bool(enable))))

    def profile_read(self):
        """{kind: (total ms, launches)} of the decode-step launches recorded since profile(True)."""
        n = len(PROFILE_KINDS)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        self._c(lib().kvo_profile_read(self.ctx, ms, cnt, n))
        return {k: (ms[i], cnt[i]) for i, k in enumerate(PROFILE_KINDS)}

    def profile_trace(self):
        """[(kind, layer, start_ms, end_ms)] of the recorded launches (before profile_read)."""
        n = ctypes.c_int(0)
        self._c(lib().kvo_profile_trace(self.ctx, None, None, None, None, 0, ctypes.byref(n)))
        m = n.value
        t0, t1 = (ctypes.c_double * m)(), (ctypes.c_double * m)()
        kd, ly = (ctypes.c_int32 * m)(), (ctypes.c_int32 * m)()
        self._c(lib().kvo_profile_trace(self.ctx, t0, t1, kd, ly, m, ctypes.byref(n)))
        return [(PROFILE_KINDS[kd[i]], ly[i], t0[i], t1[i]) for i in range(m)]

    def landmarks(self, layer, stream=None):
        C = self.info()["C_max"]
        dt = torch.float32 if self.block_size > 1 else torch.bfloat16
        dst = torch.empty(self.G, C, self.head_dim, dtype=dt, device="cuda")
        self._c(lib().kvo_landmarks(self.ctx, layer, _ptr(dst), _stream(stream)))
        return dst

    def buffer_views(self, buf):
        """(K, V) zero-copy views of ping-pong half ``buf`` as bf16 CUDA tensors [G][2k][B][d]."""
        kp, vp = ctypes.c_void_p(), ctypes.c_void_p()
        self._c(lib().kvo_buffer(self.ctx, buf, ctypes.byref(kp), ctypes.byref(vp)))
        n = self.G * 2 * self.top_k * self.block_size * self.head_dim
        return tuple(_device_view(p.value, n).view(self.G, 2 * self.top_k, self.block_size, self.head_dim)
                     for p in (kp, vp))

    def buffer(self, buf):
        """(K, V) copies of ping-pong half ``buf`` as bf16 CUDA tensors [G][2k][B][d]."""
        kp, vp = ctypes.c_void_p(), ctypes.c_void_p()
        self._c(lib().kvo_buffer(self.ctx, buf, ctypes.byref(kp), ctypes.byref(vp)))
        n = self.G * 2 * self.top_k * self.block_size * self.head_dim
        torch.cuda.synchronize()
        return tuple(_device_view(p.value, n).clone().view(self.G, 2 * self.top_k, self.block_size, self.head_dim)
                     for p in (kp, vp))


class _CudaArray:
    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i2", "data": (ptr, False), "version": 2}


def _device_view(ptr: int, n: int) -> torch.Tensor:
    """bf16 view of n library-owned device elements (no copy)."""
    return torch.as_tensor(_CudaArray(ptr, n), device="cuda").view(torch.bfloat16)
