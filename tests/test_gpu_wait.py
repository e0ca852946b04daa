"""The bounded waits of the TMA-staged attention kernel, made to run out.

The test switch (kvo_set_wait_test) makes the first warp of CTA 0 announce one
tile of its ring without copying it, so the wait for it can never complete.  The wait must give
up after the limit (here 50 ms), set KVO_DEV_TIMEOUT in the device status word
and let the kernel return, with every copy it did issue landed -- and the
context must stay usable: the same call afterwards, with the switch off, matches
the oracle.  Nothing faults or hangs: the only missing piece is a copy that is
never issued."""
import time

import pytest
import torch

from sparse_kv_cache_landmark_gb300 import kvo, synth
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close
from tests.margins import find_attempts

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("impl,skip_tile", [(1, 0), (1, 3), (2, 0), (2, 3)])
def test_attention_wait_runs_out_and_context_survives(impl, skip_tile):
    w = Workload("wait_test", 2, 8, 2, 128, 16, 24, 80, 1, (1104, 1104))
    seed = 5
    lens = synth.seq_lens(w, seed)
    groups = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    att = find_attempts(w, seed, 0, lens, lambda b, g, qr: synth.gen_request_kv(w, seed, 0, b, lens[b], qr)[0][g],
                        groups)
    c = Case(w, seed, attempts=att, gen_device="cpu")
    try:
        ctx = c.ctx
        q = c.q_dev(0)
        T, _ = ctx.select_topk(0, q)
        miss, cnt, slot = ctx.index_diff(T, None)
        ctx.gather_coalesced(0, 0, miss, cnt, slot_base=w.top_k, urgent=True)
        # two CTAs (impl 1), or two per group (impl 2: CTA 0's cluster partner
        # waits for it at the cluster barriers), so the first warp of CTA 0 has
        # several tiles and both skip positions exist
        ctx.set_attn_impl(impl, 2)
        assert ctx.device_status() == 0
        ctx.set_wait_test(50_000_000, skip_tile)
        t0 = time.perf_counter()
        ctx.sparse_decode_attn(0, 0, q, slot)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        code = ctx.device_status()
        assert code & kvo.DEV_TIMEOUT, code
        assert elapsed < 5.0                    # the limit, not a hang
        # switch off: the context works as before
        ctx.set_wait_test(2_000_000_000, -1)
        o, lse = ctx.sparse_decode_attn(0, 0, q, slot)
        torch.cuda.synchronize()
        assert ctx.device_status() == 0
        r = w.group_size
        for b, g in groups:
            ref = c.oracle_group(0, b, g)
            rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
            assert_attn_close(o[0, rows].cpu().numpy(), ref.o)
            assert_attn_close(lse[0, rows].cpu().numpy(), ref.lse, what="lse")
    finally:
        c.ctx.set_attn_impl(2, 0)
        c.close()


def test_wait_switch_rejects_bad_limits():
    w = Workload("wait_args", 1, 8, 2, 64, 16, 4, 16, 1, (336, 336))
    c = Case(w, 1, gen_device="cpu")
    try:
        with pytest.raises(kvo.KvoError):
            c.ctx.set_wait_test(10, -1)
        with pytest.raises(kvo.KvoError):
            c.ctx.set_wait_test(2_000_000_000, -2)
    finally:
        c.close()
