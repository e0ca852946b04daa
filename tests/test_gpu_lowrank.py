"""Low-rank key reconstruction of missed blocks (kvo_set_lowrank_keys) against
the oracle: the rebuilt K rows and the fetched V rows of every miss slot equal
the host rows bit for bit, and attention stays within the tolerance, in the
ping-pong and the resident buffer modes."""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import Case, assert_attn_close
from tests.margins import find_attempts

pytestmark = pytest.mark.gpu


def _workload(L, B=16, k=16):
    n = 32 + B * 64
    return Workload(f"lowrank_L{L}", 2, 8, 2, 128, B, k, 32, L, (n, n), key_dist="lowrank", lowrank_rank=32,
                    spec_sigma=0.3)


def _case(w, seed, resident=False):
    lens = synth.seq_lens(w, seed)
    groups = [(b, g) for b in range(w.batch) for g in range(w.n_kv_heads)]
    att = [find_attempts(w, seed, l, lens,
                         lambda b, g, qr, l=l: synth.gen_request_kv(w, seed, l, b, lens[b], qr)[0][g], groups)
           for l in range(w.n_layers)]
    return Case(w, seed, attempts=att, gen_device="cpu", resident=resident)


def _factors(c, layer):
    w = c.w
    R = w.lowrank_rank
    coef = torch.empty(sum(c.lens) * w.n_kv_heads * R, dtype=torch.bfloat16)
    basis = torch.empty(w.batch * w.n_kv_heads * R * w.head_dim, dtype=torch.bfloat16)
    synth.fill_lowrank(w, c.seed, layer, coef, basis, c.lens)
    return coef.cuda(), basis.cuda()


def _check_attention(c, o, lse):
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


def test_pingpong_misses_rebuilt_bit_exact():
    w = _workload(2)
    c = _case(w, 77)
    try:
        coef, basis = _factors(c, 0)
        c.ctx.set_lowrank_keys(0, w.lowrank_rank, coef, basis)      # layer 0 rebuilds, layer 1 fetches
        q, qs = c.q_stack(), c.q_stack(spec=True)
        k, B = w.top_k, w.block_size
        for step in range(3):
            o, lse = c.ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            _check_attention(c, o, lse)
            prof_miss = 0
            for l in range(2):                 # two layers: layer l always uses half l
                bk, bv = c.ctx.buffer(l)
                bk, bv = synth.bits(bk.cpu()), synth.bits(bv.cpu())
                for b in range(w.batch):
                    for g in range(w.n_kv_heads):
                        i = b * w.n_kv_heads + g
                        ref = c.oracle_group(l, b, g)
                        M = ref.T if step == 0 else ref.M          # cold step: everything is a miss
                        kr, vr = synth.bits(c.rows(l, b, g, "k")), synth.bits(c.rows(l, b, g, "v"))
                        for j, x in enumerate(M):
                            assert np.array_equal(bk[i, k + j], kr[x * B:(x + 1) * B]), (step, l, b, g, j)
                            assert np.array_equal(bv[i, k + j], vr[x * B:(x + 1) * B]), (step, l, b, g, j)
                        prof_miss += len(M)
            assert prof_miss > 0
        # and the rebuilt rows are the oracle's own low-rank keys
        R = w.lowrank_rank
        cf = synth.bits(coef.cpu()).reshape(-1, R)
        bs = synth.bits(basis.cpu()).reshape(w.batch, w.n_kv_heads, R, w.head_dim)
        off = 0
        for b in range(w.batch):
            for g in range(w.n_kv_heads):
                n = c.lens[b]
                keys = orc.lowrank_keys(cf[off:off + n], bs[b, g])
                assert np.array_equal(keys, synth.bits(c.rows(0, b, g, "k")))
                off += n
    finally:
        c.close()


def test_resident_misses_rebuilt_bit_exact():
    w = _workload(1)
    c = _case(w, 78, resident=True)
    try:
        coef, basis = _factors(c, 0)
        c.ctx.set_lowrank_keys(0, w.lowrank_rank, coef, basis)
        q, qs = c.q_stack(), c.q_stack(spec=True)
        B = w.block_size
        for step in range(3):
            o, lse = c.ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            assert c.ctx.device_status() == 0
            _check_attention(c, o, lse)
        table = c.ctx.resident_slots(0).numpy()
        bk, bv = c.ctx.buffer(2)
        bk, bv = synth.bits(bk.cpu()), synth.bits(bv.cpu())
        for b in range(w.batch):
            for g in range(w.n_kv_heads):
                i = b * w.n_kv_heads + g
                kr, vr = synth.bits(c.rows(0, b, g, "k")), synth.bits(c.rows(0, b, g, "v"))
                for sl, x in enumerate(table[i].tolist()):
                    if x >= 0:
                        assert np.array_equal(bk[i, sl], kr[x * B:(x + 1) * B])
                        assert np.array_equal(bv[i, sl], vr[x * B:(x + 1) * B])
    finally:
        c.close()


def test_lowrank_arguments_are_checked():
    w = _workload(1)
    c = _case(w, 79)
    try:
        with pytest.raises(Exception, match="rank"):
            c.ctx.set_lowrank_keys(0, 65, None, None)
        with pytest.raises(Exception, match="coef"):
            c.ctx.set_lowrank_keys(0, 32, None, None)
        c.ctx.set_lowrank_keys(0, 0, None, None)            # off again
    finally:
        c.close()
