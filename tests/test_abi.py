"""The C ABI library: builds, loads, exports every declared symbol, and
rejects bad arguments on the host before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvo.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_cache_landmark_gb300 import build, kvo
    build.build()
    return kvo.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["kv_offload_init", "select_topk", "index_diff", "gather_coalesced", "sparse_decode_attn", "merge_lse"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_binding_names_match_header():
    from sparse_kv_cache_landmark_gb300 import kvo
    assert sorted(kvo.EXPORTS) == declared_functions()


def _cfg(kvo, **kw):
    base = dict(batch=1, n_q_heads=8, n_kv_heads=2, head_dim=64, block_size=16, top_k=4, window=16, n_layers=1)
    base.update(kw)
    lens = (ctypes.c_int32 * max(base["batch"], 1))(*([16 * 20 + 16] * max(base["batch"], 1)))
    return kvo._Config(base["batch"], base["n_q_heads"], base["n_kv_heads"], base["head_dim"], base["block_size"],
                       base["top_k"], base["window"], base["n_layers"], lens, base.get("max_append", 0)), lens


@pytest.mark.parametrize("kw,frag", [
    (dict(batch=0), "batch"),
    (dict(n_q_heads=7), "head"),
    (dict(n_q_heads=64, n_kv_heads=2), "<= 16"),
    (dict(head_dim=96), "head_dim"),
    (dict(top_k=0), "top_k"),
    (dict(top_k=21), "top_k exceeds"),
    (dict(block_size=7), "block_size == 0"),
    (dict(max_append=-1), "max_append"),
    (dict(max_append=8, window=24), "window % block_size"),
])
def test_init_rejects_bad_configs_on_the_host(lib, kw, frag):
    from sparse_kv_cache_landmark_gb300 import kvo
    cfg, lens = _cfg(kvo, **kw)
    dummy = (ctypes.c_void_p * 1)(1)
    out = ctypes.c_void_p()
    st = lib.kv_offload_init(ctypes.byref(cfg), dummy, dummy, dummy, dummy, ctypes.byref(out))
    assert st == kvo.KVO_ERR_INVALID
    assert out.value is None
    assert frag in lib.kvo_last_error(None).decode()


def test_null_arguments_are_rejected(lib):
    from sparse_kv_cache_landmark_gb300 import kvo
    out = ctypes.c_void_p()
    assert lib.kv_offload_init(None, None, None, None, None, ctypes.byref(out)) == kvo.KVO_ERR_INVALID
    assert lib.kv_offload_init(None, None, None, None, None, None) == kvo.KVO_ERR_INVALID
    assert lib.select_topk(None, 0, None, None, None, None, None) == kvo.KVO_ERR_INVALID
    assert lib.merge_lse(None, None, None, None, None, None, -1, 4, None) == kvo.KVO_ERR_INVALID
    assert lib.merge_lse(None, None, None, None, None, None, 3, 4, None) == kvo.KVO_ERR_INVALID
    assert lib.kvo_set_select_impl(None, 1) == kvo.KVO_ERR_INVALID
    assert lib.kvo_set_attn_impl(None, 2, 0) == kvo.KVO_ERR_INVALID
    assert lib.kv_offload_destroy(None) == kvo.KVO_OK
    assert lib.merge_lse(None, None, None, None, None, None, 0, 4, None) == kvo.KVO_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from sparse_kv_cache_landmark_gb300 import kvo
    monkeypatch.setattr(kvo, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(kvo, "_LIB", None)
    with pytest.raises(RuntimeError, match="not built"):
        kvo.lib()


def test_static_attention_wrapper_checks_every_buffer():
    """sparse_decode_attn_static has no context to size its buffers by: the
    binding checks dtype, contiguity, size and device of each one before the
    call, so a short buffer never reaches the GPU (no library call is made)."""
    import torch
    from sparse_kv_cache_landmark_gb300 import kvo
    shape = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=64, block_size=16, top_k=4, window=16)
    G, rows = 4, 16
    bf = lambda n: torch.zeros(n, dtype=torch.bfloat16)
    q, kb, vb = bf(rows * 64), bf(G * 8 * 16 * 64), bf(G * 8 * 16 * 64)
    slot = torch.zeros(G * 4, dtype=torch.int32)
    kw, vw = bf(G * 16 * 64), bf(G * 16 * 64)
    call = lambda **over: kvo.sparse_decode_attn_static(
        *[over.get(n, t) for n, t in (("q", q), ("k_buf", kb), ("v_buf", vb), ("slot", slot), ("k_win", kw),
                                      ("v_win", vw))], **{**shape, **over.get("shape", {})},
        **{k: v for k, v in over.items() if k in ("o", "lse", "status")})
    with pytest.raises(kvo.KvoError, match="k_buf holds"):
        call(k_buf=bf(G * 8 * 16 * 64 - 1))
    with pytest.raises(kvo.KvoError, match="slot_of_true must be torch.int32"):
        call(slot=slot.long())
    with pytest.raises(kvo.KvoError, match="v_win holds"):
        call(v_win=bf(10))
    with pytest.raises(kvo.KvoError, match="k_win is required"):
        call(k_win=None)
    with pytest.raises(kvo.KvoError, match="contiguous"):
        call(q=bf(2 * rows * 64)[::2])
    with pytest.raises(kvo.KvoError, match="o holds"):
        call(o=torch.zeros(5, dtype=torch.float32))
    with pytest.raises(kvo.KvoError, match="status must be torch.int32"):
        call(status=torch.zeros(1, dtype=torch.float32))
    # right sizes on the CPU: rejected for the device, still before any library call
    with pytest.raises(kvo.KvoError, match="one CUDA device"):
        call()
    # no window: the window buffers may be None
    with pytest.raises(kvo.KvoError, match="one CUDA device"):
        call(k_win=None, v_win=None, shape=dict(window=0))
