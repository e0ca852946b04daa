"""sparse_decode_attn_static: the context-free attention call whose scratch is
a static device array, for callers that cannot allocate device memory (their
memory belongs to another allocator, or a decode loop cannot afford the
implicit synchronisation of cudaMalloc / cudaFree).  Checked through the C ABI
against sparse_decode_attn on the same inputs, on two calls in a row.  This
file is collected last so that a run stopping at the first failure has run
every other test first."""
import pytest
import torch

from sparse_kv_cache_landmark_gb300 import kvo
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fuse", [True, False])
def test_static_scratch_attention_matches_context_call(fuse):
    w = Workload("no_alloc", 3, 8, 2, 128, 16, 24, 80, 1, (1104, 2128), spec_sigma=0.3)
    c = Case(w, 31, gen_device="cpu")
    try:
        ctx = c.ctx
        q = c.q_dev(0)
        T, P = ctx.select_topk(0, q, c.q_dev(0, spec=True))
        miss, cnt, slot = ctx.index_diff(T, P)
        ctx.gather_coalesced(0, 1, P, None, slot_base=0)
        ctx.gather_coalesced(0, 1, miss, cnt, slot_base=w.top_k, urgent=True)
        ref_o, ref_lse = ctx.sparse_decode_attn(0, 1, q, slot, fuse_window_merge=fuse)
        kb, vb = ctx.buffer_views(1)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = dict(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                    block_size=w.block_size, top_k=w.top_k, window=w.window, fuse_window_merge=fuse,
                    status=status)
        for _ in range(2):
            o, lse = kvo.sparse_decode_attn_static(q, kb, vb, slot, c.k_win[0], c.v_win[0], **args)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert_attn_close(o.cpu().numpy(), ref_o.cpu().numpy())
            assert_attn_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), what="lse")
        assert ctx.device_status() == 0
    finally:
        c.close()


def test_static_scratch_rejects_oversized_calls():
    q = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kvo.KvoError, match="static scratch"):
        kvo.sparse_decode_attn_static(q, q, q, i, q, q, batch=512, n_q_heads=128, n_kv_heads=8, head_dim=128,
                                      block_size=64, top_k=8192, window=512)
