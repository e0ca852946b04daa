"""The pipelined multi-layer decode step (prefetch two layers ahead into the
ping-pong buffer, urgent misses, attention) against the oracle, cold and warm,
for odd, even and single-layer models, with and without speculation."""
import numpy as np
import pytest
import torch

from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close
from tests.margins import find_attempts

pytestmark = pytest.mark.gpu


def _case(L, spec, seed=4242):
    w = Workload(f"step_L{L}", 2, 8, 2, 128, 16, 16, 32, L, (1056, 1056), spec_sigma=0.3 if spec else None)
    lens = synth.seq_lens(w, seed)
    groups = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    att = [find_attempts(w, seed, l, lens,
                         lambda b, g, qr, l=l: synth.gen_request_kv(w, seed, l, b, lens[b], qr)[0][g], groups)
           for l in range(L)]
    return Case(w, seed, attempts=att, gen_device="cpu")


def _check(c, o, lse):
    w = c.w
    r = w.group_size
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    for l in range(c.L):
        for b in range(w.batch):
            for g in range(w.n_kv_heads):
                ref = c.oracle_group(l, b, g)
                rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                assert_attn_close(o[l, rows], ref.o, what=f"o layer {l}")
                assert_attn_close(lse[l, rows], ref.lse, what=f"lse layer {l}")


@pytest.mark.parametrize("L,spec", [(1, True), (4, True), (5, True), (3, False), (2, False)])
def test_decode_step_cold_and_warm(L, spec):
    c = _case(L, spec)
    try:
        q = c.q_stack()
        qs = c.q_stack(spec=True)
        outs = []
        for step in range(3):
            o, lse = c.ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            _check(c, o, lse)
            outs.append((o.clone(), lse.clone()))
        # the prediction never changes the result (DualDecoder: attention over the
        # miss-corrected buffer equals attention over the true selection)
        for o, lse in outs[1:]:
            np.testing.assert_allclose(o.cpu().numpy(), outs[0][0].cpu().numpy(), rtol=1e-5, atol=1e-5)
        c.ctx.reset_prediction()
        o, lse = c.ctx.decode_step(q, qs)
        torch.cuda.synchronize()
        _check(c, o, lse)
    finally:
        c.close()


def test_decode_step_profile_counts_launches():
    c = _case(4, True)
    try:
        q, qs = c.q_stack(), c.q_stack(spec=True)
        c.ctx.decode_step(q, qs)
        c.ctx.profile(True)
        c.ctx.decode_step(q, qs)
        prof = c.ctx.profile_read()
        c.ctx.profile(False)
        L = c.L
        assert prof["select"][1] == L and prof["diff"][1] == L and prof["attention"][1] == L
        assert prof["gather_urgent"][1] == L and prof["gather_prefetch"][1] == L
        assert prof["coalesce"][1] == 2 * L
        assert all(ms >= 0 for ms, _ in prof.values())
    finally:
        c.close()
