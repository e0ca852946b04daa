"""Builds contexts on the GPU from seeded workloads and runs the oracle on
chosen groups.  Shared by the GPU tests, the smoke entry and nothing else."""
import numpy as np
import torch

import oracle as orc
from sparse_kv_cache_landmark_gb300 import synth
from sparse_kv_cache_landmark_gb300.kvo import Context


class Case:
    """Host caches (pinned), windows (device), queries and a library context."""

    def __init__(self, w, seed, attempts=None, n_layers=None, gen_device="cuda", resident=False):
        self.w, self.seed = w, seed
        self.L = n_layers or w.n_layers
        self.lens = synth.seq_lens(w, seed)
        n = synth.layer_numel(w, self.lens)
        self.attempts = attempts
        self.q, self.qs = [], []
        self.k_host, self.v_host, self.k_win, self.v_win = [], [], [], []
        per_layer = isinstance(attempts, (list, tuple))
        for l in range(self.L):
            a = (attempts[l] if per_layer else (attempts if l == 0 else None))
            q, qs = synth.gen_queries(w, seed, l, a)
            kh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
            vh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
            synth.fill_layer(w, seed, l, kh, vh, q, self.lens, device=gen_device)
            self.q.append(q); self.qs.append(qs)
            self.k_host.append(kh); self.v_host.append(vh)
            self.k_win.append(self._window(kh)); self.v_win.append(self._window(vh))
        self.ctx = Context(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                           block_size=w.block_size, top_k=w.top_k, window=w.window, n_layers=self.L,
                           seq_lens=self.lens, k_host=self.k_host, v_host=self.v_host,
                           k_win=self.k_win if w.window > 0 else None, v_win=self.v_win if w.window > 0 else None,
                           resident=resident)

    def _window(self, host):
        w = self.w
        out = torch.empty(w.batch, w.n_kv_heads, max(w.window, 1), w.head_dim, dtype=torch.bfloat16, device="cuda")
        off = 0
        for b, n in enumerate(self.lens):
            req = host[off:off + n * w.n_kv_heads * w.head_dim].view(w.n_kv_heads, n, w.head_dim)
            if w.window:
                out[b] = req[:, n - w.window:, :].to("cuda")
            off += n * w.n_kv_heads * w.head_dim
        return out

    def rows(self, layer, b, g, kv="k"):
        """Group rows [len_b][d] as a CPU bf16 tensor view of the host cache."""
        w = self.w
        host = (self.k_host if kv == "k" else self.v_host)[layer]
        off = sum(self.lens[:b]) * w.n_kv_heads * w.head_dim + g * self.lens[b] * w.head_dim
        return host[off: off + self.lens[b] * w.head_dim].view(self.lens[b], w.head_dim)

    def q_stack(self, spec=False):
        """All layers' queries as one device tensor [L][b][Hq][d] (None without speculation)."""
        ts = self.qs if spec else self.q
        if ts[0] is None:
            return None
        return torch.stack(ts).to("cuda").contiguous()

    def q_dev(self, layer, spec=False):
        t = (self.qs if spec else self.q)[layer]
        return None if t is None else t.to("cuda").contiguous()

    def oracle_group(self, layer, b, g, prediction=None, with_spec=True):
        w = self.w
        r = w.group_size
        qg = synth.bits(self.q[layer][b, g * r:(g + 1) * r])
        qs = self.qs[layer]
        qsg = synth.bits(qs[b, g * r:(g + 1) * r]) if (qs is not None and with_spec) else None
        return orc.decode_group(synth.bits(self.rows(layer, b, g, "k")), synth.bits(self.rows(layer, b, g, "v")),
                                qg, qsg, block_size=w.block_size, top_k=w.top_k, window=w.window,
                                prediction=prediction)

    def close(self):
        self.ctx.close()


def assert_attn_close(got, ref, atol=1e-2, rtol=1e-2, what="o"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    same = got == ref                      # equal values, including equal infinities (an empty part's lse)
    with np.errstate(invalid="ignore"):
        err = np.where(same, 0.0, np.abs(got - ref))
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)                  # NaN in either never passes
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside {atol}+{rtol}|ref|; max err {err.max():.3e}"
