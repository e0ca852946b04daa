"""Growing the cache (kvo_append): every appended token joins the GPU window;
full blocks leave it for the host cache and become candidates with a landmark.
After each append, the decode step must match the oracle run on the grown
cache (candidates [0, C*B), window [C*B, len))."""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.kvo import Context
from sparse_kv_cache_landmark_gb300.workloads import Workload
from tests.harness import assert_attn_close
from tests.margins import MARGIN

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,spec,L,att,resident", [(16, True, 2, (1, 0), False), (1, False, 1, (1, 0), False),
                                                   (32, False, 3, (1, 0), False), (16, False, 1, (0, 0), False),
                                                   (16, False, 1, (1, 2), False), (16, True, 2, (1, 0), True),
                                                   (16, True, 2, (2, 3), False), (16, False, 2, (2, 0), True)])
def test_append_grows_the_cache(B, spec, L, att, resident):
    W, n_app, d = 32, 40 if B > 1 else 12, 128
    len0 = W + B * 20 if B > 1 else W + 400
    cap = len0 + n_app
    w = Workload(f"append_B{B}", 2, 8, 2, d, B, 8, W, L, (cap, cap), spec_sigma=0.3 if spec else None)
    seed = 55
    lens_full = synth.seq_lens(w, seed)
    G, r = w.batch * w.n_kv_heads, w.group_size
    full = [synth.make_layer(w, seed, layer=l) for l in range(L)]         # all cap tokens of every group
    k_host, v_host, k_win, v_win = [], [], [], []
    for l in range(L):
        kh = full[l].k.clone().pin_memory()
        vh = full[l].v.clone().pin_memory()
        khv = kh.view(w.batch, w.n_kv_heads, cap, d)
        vhv = vh.view(w.batch, w.n_kv_heads, cap, d)
        khv[:, :, len0:] = 0                 # spare capacity: kvo_append must fill it
        vhv[:, :, len0:] = 0
        k_host.append(kh); v_host.append(vh)
        k_win.append(khv[:, :, len0 - W:len0].contiguous().cuda())
        v_win.append(vhv[:, :, len0 - W:len0].contiguous().cuda())
    ctx = Context(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=d, block_size=B,
                  top_k=w.top_k, window=W, n_layers=L, seq_lens=[len0] * w.batch, k_host=k_host, v_host=v_host,
                  k_win=k_win, v_win=v_win, max_append=n_app, resident=resident)
    try:
        ctx.set_attn_impl(*att)        # the window ring wraps inside and across attention tiles
        q = torch.stack([full[l].q for l in range(L)]).cuda()
        qs = torch.stack([full[l].q_spec for l in range(L)]).cuda() if spec else None
        checked = skipped = 0
        for j in range(n_app + 1):
            n = len0 + j
            C = (n - W) // B
            wn = n - C * B                        # window between W and W + B - 1 tokens
            o, lse = ctx.decode_step(q, qs)
            torch.cuda.synchronize()
            assert ctx.device_status() == 0
            on, ln = o.cpu().numpy(), lse.cpu().numpy()
            for l in range(L):
                fk = synth.bits(full[l].k).reshape(w.batch, w.n_kv_heads, cap, d)
                fv = synth.bits(full[l].v).reshape(w.batch, w.n_kv_heads, cap, d)
                for b in range(w.batch):
                    for g in range(w.n_kv_heads):
                        qg = synth.bits(full[l].q[b, g * r:(g + 1) * r])
                        ref = orc.decode_group(fk[b, g, :n], fv[b, g, :n], qg, None, block_size=B,
                                               top_k=w.top_k, window=wn)
                        if orc.kth_relative_gap(ref.scores_true, w.top_k) < MARGIN:
                            skipped += 1
                            continue
                        rows = slice(b * w.n_q_heads + g * r, b * w.n_q_heads + (g + 1) * r)
                        assert_attn_close(on[l, rows], ref.o, what=f"o after {j} appends")
                        assert_attn_close(ln[l, rows], ref.lse, what=f"lse after {j} appends")
                        checked += 1
            if j == n_app:
                break
            kn = torch.stack([full[l].k.view(w.batch, w.n_kv_heads, cap, d)[:, :, n] for l in range(L)]).cuda()
            vn = torch.stack([full[l].v.view(w.batch, w.n_kv_heads, cap, d)[:, :, n] for l in range(L)]).cuda()
            ctx.append(kn.contiguous(), vn.contiguous())
        assert checked > 3 * skipped
        # evicted blocks were written to the host cache, bit for bit, and gained landmarks
        n = len0 + n_app
        C = (n - W) // B
        C0 = (len0 - W) // B
        assert C > C0
        for l in range(L):
            got = synth.bits(k_host[l]).reshape(w.batch, w.n_kv_heads, cap, d)
            exp = synth.bits(full[l].k).reshape(w.batch, w.n_kv_heads, cap, d)
            assert np.array_equal(got[:, :, :C * B], exp[:, :, :C * B])
            # rows past both the evicted blocks and the initial cache are still untouched
            assert not got[:, :, max(C * B, len0):].any()
            gv = synth.bits(v_host[l]).reshape(w.batch, w.n_kv_heads, cap, d)
            ev = synth.bits(full[l].v).reshape(w.batch, w.n_kv_heads, cap, d)
            assert np.array_equal(gv[:, :, :C * B], ev[:, :, :C * B])
            lm = ctx.landmarks(l).cpu()
            for b in range(w.batch):
                for g in range(w.n_kv_heads):
                    ref = orc.landmarks(exp[b, g, :C * B], B, C)
                    np.testing.assert_allclose(lm[b * w.n_kv_heads + g, :C].double().numpy(), ref,
                                               rtol=2e-6, atol=1e-7)
        with pytest.raises(Exception, match="capacity"):
            ctx.append(kn.contiguous(), vn.contiguous())
    finally:
        ctx.close()
