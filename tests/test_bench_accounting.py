"""The benchmark's algorithmic byte counts (the numerators of its rooflines)
against closed forms of the step's traffic.

Per layer and step the step reads the landmarks once (C blocks x d fp32 per
KV head), writes the k gathered blocks of every group, reads them and the W
window tokens back in attention, and moves the gathered blocks over the host
link; a resident step moves only the blocks it fetched, and a low-rank layer
moves only the values of its misses.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_kv_cache_landmark_gb300.workloads import WORKLOADS  # noqa: E402


def test_llama_shape_bytes():
    w = WORKLOADS["llama3_8b_decode"]
    lens = [32768] * w.batch
    by = bench.workload_bytes(w, lens)
    # 16 requests x 8 KV heads, 64 blocks of 32 tokens, 512 B of K+V per token, 32 layers
    assert by["host"] == 16 * 8 * 64 * 32 * 512 * 32 == 4_294_967_296
    assert by["gather_per_launch"] == 16 * 8 * 64 * 32 * 512 == 134_217_728
    # attention reads the 2048 gathered tokens and the 512 window tokens of every group
    assert by["attended_per_layer"] == 16 * 8 * (64 * 32 + 512) * 512 == 167_772_160
    assert by["kv_attended"] == by["attended_per_layer"] * 32
    # fp32 landmarks: (32768 - 512) / 32 = 1008 blocks per request and KV head
    assert by["landmark_per_layer"] == 16 * 1008 * 8 * 128 * 4
    # HBM: landmarks + gathered writes + attended reads dominate (q, o/lse, index lists are small)
    big = (by["landmark_per_layer"] + by["gather_per_launch"] + by["attended_per_layer"]) * 32
    assert big < by["hbm"] < big * 1.01
    assert by["urgent"] == 0


def test_misses_add_urgent_bytes():
    w = WORKLOADS["long_ctx_predict"]
    lens = [65536 + 32 * i for i in range(w.batch)]
    base = bench.workload_bytes(w, lens)
    with_m = bench.workload_bytes(w, lens, misses_per_step=1000)
    one_block = w.block_size * 4 * w.head_dim
    assert with_m["host"] - base["host"] == 1000 * one_block
    assert with_m["hbm"] - base["hbm"] == 1000 * one_block
    # ragged lengths: the landmark bytes follow each request's own block count
    C = [(n - w.window) // w.block_size for n in lens]
    assert base["landmark_per_layer"] == sum(C) * w.n_kv_heads * w.head_dim * 4


def test_resident_and_lowrank_bytes():
    w = WORKLOADS["llama3_8b_decode"]
    lens = [32768] * w.batch
    one_block = w.block_size * 4 * w.head_dim
    res = bench.workload_bytes(w, lens, fetched_per_step=12744)
    # only the fetched blocks cross the link; nothing else is gathered
    assert res["host"] == 12744 * one_block
    full = bench.workload_bytes(w, lens)
    assert full["hbm"] - res["hbm"] == full["gather_per_launch"] * 32 - 12744 * one_block
    # low-rank keys: misses move V only, and the rebuild reads R bf16 coefficients per token
    lw = WORKLOADS["lowrank_predict"]
    llens = [lw.ctx[0]] * lw.batch
    plain = bench.workload_bytes(lw, llens, misses_per_step=100)
    rec = bench.workload_bytes(lw, llens, misses_per_step=100, recon_rank=32)
    half = 100 * lw.block_size * 2 * lw.head_dim
    assert plain["host"] - rec["host"] == half
    assert rec["hbm"] - plain["hbm"] == 100 * lw.block_size * 32 * 2
