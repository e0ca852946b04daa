"""Calls of different scratch classes on one context may overlap on the GPU.

Selection (its keys, histograms and tickets) and attention (its work items,
partials and tickets) use disjoint context scratch, so a caller may run the
selection, diff and gather of layer l + 1 on one stream while the attention
of layer l runs on another -- the overlap a layer-pipelined caller wants.
Two attention calls, or two selections, are ordered on one stream (or by an
event) instead.  Both layers' indices and outputs must match the oracle."""
import numpy as np
import pytest
import torch

from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close
from tests.margins import find_attempts

pytestmark = pytest.mark.gpu


def test_selection_and_attention_overlap_on_two_streams():
    w = Workload("two_streams", 3, 8, 2, 128, 16, 24, 80, 2, (1104, 2128))
    seed = 41
    lens = synth.seq_lens(w, seed)
    groups = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    att = [find_attempts(w, seed, l, lens,
                         lambda b, g, qr, l=l: synth.gen_request_kv(w, seed, l, b, lens[b], qr)[0][g], groups)
           for l in range(2)]
    c = Case(w, seed, attempts=att, gen_device="cpu")
    try:
        ctx, k = c.ctx, w.top_k
        q = [c.q_dev(l) for l in range(2)]
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        # stream A: layer 0's index and urgent gather into half 0
        T0, _ = ctx.select_topk(0, q[0], stream=sa)
        m0, c0, slot0 = ctx.index_diff(T0, None, stream=sa)
        ctx.gather_coalesced(0, 0, m0, c0, slot_base=k, urgent=True, stream=sa)
        ready0 = torch.cuda.Event()
        ready0.record(sa)
        # stream B: layer 0's attention once its blocks are in ...
        sb.wait_event(ready0)
        o0, l0 = ctx.sparse_decode_attn(0, 0, q[0], slot0, stream=sb)
        done0 = torch.cuda.Event()
        done0.record(sb)
        # ... while stream A selects and gathers layer 1 into half 1
        T1, _ = ctx.select_topk(1, q[1], stream=sa)
        m1, c1, slot1 = ctx.index_diff(T1, None, stream=sa)
        ctx.gather_coalesced(1, 1, m1, c1, slot_base=k, urgent=True, stream=sa)
        # the second attention call is ordered after the first (same scratch class)
        sa.wait_event(done0)
        o1, l1 = ctx.sparse_decode_attn(1, 1, q[1], slot1, stream=sa)
        torch.cuda.synchronize()
        assert ctx.device_status() == 0
        r = w.group_size
        for layer, T, o, lse in ((0, T0, o0, l0), (1, T1, o1, l1)):
            T, o, lse = T.cpu(), o.cpu().numpy(), lse.cpu().numpy()
            for b, g in groups:
                ref = c.oracle_group(layer, b, g)
                assert T[b * w.n_kv_heads + g].tolist() == ref.T.tolist(), (layer, b, g)
                rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                assert_attn_close(o[0, rows], ref.o)
                assert_attn_close(lse[0, rows], ref.lse, what="lse")
        assert not np.array_equal(T0.cpu().numpy(), T1.cpu().numpy())   # two distinct layers were served
    finally:
        c.close()
