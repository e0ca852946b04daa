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


@pytest.mark.parametrize("L,spec,engine", [(1, True, 3), (4, True, 3), (5, True, 3), (3, False, 3), (2, False, 3),
                                           (4, True, 0), (1, True, 0), (3, False, 0),
                                           (4, True, 1), (1, True, 1)])
def test_decode_step_cold_and_warm(L, spec, engine):
    c = _case(L, spec)
    try:
        c.ctx.set_gather_engine(engine, 4 if engine == 1 else 0)
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


def test_decode_step_attention_kernels_agree():
    """The decode step matches the oracle with any attention kernel, TMA grid
    or cluster split (the kernels split tiles differently: equal up to
    rounding)."""
    c = _case(4, True)
    try:
        q, qs = c.q_stack(), c.q_stack(spec=True)
        res = []
        for impl, ctas in ((1, 0), (0, 0), (1, 2), (2, 0), (2, 3)):
            c.ctx.set_attn_impl(impl, ctas)
            for _ in range(2):
                o, lse = c.ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            res.append((o.cpu(), lse.cpu()))
        for o, lse in res:
            _check(c, o, lse)
            np.testing.assert_allclose(o.numpy(), res[0][0].numpy(), rtol=1e-2, atol=2e-3)
    finally:
        c.close()


@pytest.mark.parametrize("engine", [3, 0])
def test_decode_step_profile_counts_launches(engine):
    c = _case(4, True)
    try:
        c.ctx.set_gather_engine(engine, 0)
        q, qs = c.q_stack(), c.q_stack(spec=True)
        c.ctx.decode_step(q, qs)
        c.ctx.profile(True)
        c.ctx.decode_step(q, qs)
        trace = c.ctx.profile_trace()
        prof = c.ctx.profile_read()
        c.ctx.profile(False)
        L = c.L
        assert prof["select"][1] == L and prof["diff"][1] == L and prof["attention"][1] == L
        assert prof["gather_urgent"][1] == L and prof["gather_prefetch"][1] == L
        # the flat engine copies straight from the index lists; the others walk run lists
        assert prof["coalesce"][1] == (0 if engine == 3 else 2 * L)
        assert all(ms >= 0 for ms, _ in prof.values())
        assert len(trace) == sum(n for _, n in prof.values())
        assert all(t1 >= t0 for _, _, t0, t1 in trace)
        assert sorted({l for k, l, _, _ in trace if k == "attention"}) == list(range(L))
    finally:
        c.close()


def test_decode_step_dual_cobatched():
    c = _case(4, True)
    try:
        q, qs = c.q_stack(), c.q_stack(spec=True)
        for step in range(2):
            o, lse, os_, ls_ = c.ctx.decode_step_dual(q, qs)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            _check(c, o, lse)
            w = c.w
            r = w.group_size
            on, ln = os_.cpu().numpy(), ls_.cpu().numpy()
            for l in range(c.L):
                for b in range(w.batch):
                    for g in range(w.n_kv_heads):
                        ref = c.oracle_group(l, b, g)
                        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                        assert_attn_close(on[l, rows], ref.o_spec, what="o_spec")
                        assert_attn_close(ln[l, rows], ref.lse_spec, what="lse_spec")
    finally:
        c.close()


@pytest.mark.parametrize("L,spec,engine", [(4, True, 0), (1, True, 3), (3, False, 3)])
def test_decode_step_graph_replay(L, spec, engine):
    """Graph-replayed warm steps give the same outputs as stream-launched ones."""
    c = _case(L, spec)
    try:
        c.ctx.set_gather_engine(engine, 0)
        q, qs = c.q_stack(), c.q_stack(spec=True)
        o0, l0 = c.ctx.decode_step(q, qs)
        o1, l1 = c.ctx.decode_step(q, qs)
        ref_o, ref_l = o1.clone(), l1.clone()
        c.ctx.set_graphs(True)
        o = torch.empty_like(o1)
        lse = torch.empty_like(l1)
        for step in range(5):                 # captures parity 0 and 1, then replays
            o.fill_(float("nan"))
            c.ctx.decode_step(q, qs, o, lse)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            np.testing.assert_allclose(o.cpu().numpy(), ref_o.cpu().numpy(), rtol=1e-5, atol=1e-5)
            np.testing.assert_allclose(lse.cpu().numpy(), ref_l.cpu().numpy(), rtol=1e-5, atol=1e-5)
        _check(c, o, lse)
        c.ctx.set_graphs(False)
        for step in range(2):                 # stream-launched steps after graph steps
            o2, l2 = c.ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            np.testing.assert_allclose(o2.cpu().numpy(), ref_o.cpu().numpy(), rtol=1e-5, atol=1e-5)
        c.ctx.set_graphs(True)                # and back to graphs with new output pointers
        o3, l3 = c.ctx.decode_step(q, qs)
        o3, l3 = c.ctx.decode_step(q, qs)
        torch.cuda.synchronize()
        np.testing.assert_allclose(o3.cpu().numpy(), ref_o.cpu().numpy(), rtol=1e-5, atol=1e-5)
        assert c.ctx.device_status() == 0
    finally:
        c.close()
