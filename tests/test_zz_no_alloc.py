"""sparse_decode_attn_static: the context-free attention call whose scratch is
a static device array, for callers that cannot allocate device memory (their
memory belongs to another allocator, or a decode loop cannot afford the
implicit synchronisation of cudaMalloc / cudaFree).  Checked through the C ABI
against the fp64 oracle and against sparse_decode_attn on the same inputs, on
two calls in a row, in shapes that reach both query-row layouts (r <= 8 and
r = 16), both head dims and a cache without a window (NULL window pointers).
This file is collected last so that a run stopping at the first failure has
run every other test first."""
import ctypes

import pytest
import torch

from sparse_kv_cache_landmark_gb300 import kvo, synth
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close
from tests.margins import find_attempts

pytestmark = pytest.mark.gpu

SHAPES = {
    # d 128, r 4, ragged lengths, a window of 80 tokens
    "d128_r4": Workload("no_alloc", 3, 8, 2, 128, 16, 24, 80, 1, (1104, 2128), spec_sigma=0.3),
    # d 64, r 8, no window: the window pointers are NULL
    "d64_r8_nowin": Workload("no_alloc_nowin", 2, 16, 2, 64, 32, 8, 0, 1, (2048, 2048)),
    # r 16 fills all 16 rows of the tensor-core tiles
    "d128_r16": Workload("no_alloc_r16", 1, 32, 2, 128, 8, 32, 32, 1, (1056, 1056), key_dist="channel_scaled"),
}


def _case(w, seed):
    lens = synth.seq_lens(w, seed)
    groups = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    att = find_attempts(w, seed, 0, lens, lambda b, g, qr: synth.gen_request_kv(w, seed, 0, b, lens[b], qr)[0][g],
                        groups)
    return Case(w, seed, attempts=att, gen_device="cpu")


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("fuse", [True, False])
def test_static_scratch_attention_matches_oracle_and_context_call(shape, fuse):
    w = SHAPES[shape]
    c = _case(w, 31)
    try:
        ctx = c.ctx
        q = c.q_dev(0)
        qs = c.q_dev(0, spec=True)
        T, P = ctx.select_topk(0, q, qs)
        if P is None:
            P = T.clone()
        miss, cnt, slot = ctx.index_diff(T, P)
        ctx.gather_coalesced(0, 1, P, None, slot_base=0)
        ctx.gather_coalesced(0, 1, miss, cnt, slot_base=w.top_k, urgent=True)
        ref_o, ref_lse = ctx.sparse_decode_attn(0, 1, q, slot, fuse_window_merge=fuse)
        kb, vb = ctx.buffer_views(1)
        kw, vw = (c.k_win[0], c.v_win[0]) if w.window else (None, None)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = dict(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                    block_size=w.block_size, top_k=w.top_k, window=w.window, fuse_window_merge=fuse,
                    status=status)
        refs = {(b, g): c.oracle_group(0, b, g) for b in range(w.batch) for g in range(w.n_kv_heads)}
        r = w.group_size
        for _ in range(2):
            o, lse = kvo.sparse_decode_attn_static(q, kb, vb, slot, kw, vw, **args)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            # the context-owned call on the same buffers
            assert_attn_close(o.cpu().numpy(), ref_o.cpu().numpy())
            assert_attn_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), what="lse")
            # and the fp64 oracle, group by group
            o_np, lse_np = o.cpu().numpy(), lse.cpu().numpy()
            for (b, g), ref in refs.items():
                rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                if fuse:
                    assert_attn_close(o_np[0, rows], ref.o)
                    assert_attn_close(lse_np[0, rows], ref.lse, what="lse")
                else:
                    assert_attn_close(o_np[0, rows], ref.o_sparse, what="o_sparse")
                    assert_attn_close(lse_np[0, rows], ref.lse_sparse, what="lse_sparse")
                    if w.window:
                        assert_attn_close(o_np[1, rows], ref.o_window, what="o_window")
                        assert_attn_close(lse_np[1, rows], ref.lse_window, what="lse_window")
                    else:
                        assert (lse_np[1, rows] == -float("inf")).all() and not o_np[1, rows].any()
        assert ctx.device_status() == 0
    finally:
        c.close()


def test_static_scratch_rejects_oversized_calls():
    """The C entry point itself refuses a shape whose scratch exceeds the array
    (before touching any buffer), with both sizes in the message."""
    L = kvo.lib()
    q = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(4, dtype=torch.int32, device="cuda")
    f = torch.zeros(4, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.sparse_decode_attn_static(p(q), p(q), p(q), p(i), p(q), p(q), p(f), p(f), None, 512, 128, 8, 128, 64,
                                     8192, 512, 1, kvo._stream(None))
    assert st == kvo.KVO_ERR_INVALID
    assert "static scratch" in L.kvo_last_error(None).decode()
