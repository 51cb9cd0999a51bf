"""The run entry points inside a CUDA graph: captured once, replayed, bit for bit equal to the
eager runs. The runs allocate nothing and never synchronise, and the decode's in-kernel merge
counters return to zero after every complete run, so a captured run can be replayed ("CUDAGraph
compatible" on the FlashInfer cheat page). Each entry point is called once eagerly before the
capture (first calls look up per-device addresses)."""

import math

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth

pytestmark = pytest.mark.gpu


def _graph_equal(run, outs):
    """Eager results of run(), then a graph of run() replayed twice: equal every time."""
    run()
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    for o in outs:
        o.fill_(float("nan") if o.dtype.is_floating_point else 0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan") if o.dtype.is_floating_point else 0)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, ref):
            assert torch.equal(a, b)
    assert bskv.bskv_get_device_status() == 0


def test_graph_decode_with_in_kernel_merge(cuda):
    d = synth.paged_decode_inputs(930, 6, 32, 8, 128, 16, 1, 2000)
    p = bskv.bskv_plan_decode(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"],
                              d["num_pages"], 16, 32, 8, 128, torch.bfloat16)
    p.upload(cuda)
    assert p.metadata()[6] > 0  # split units merged inside the kernel
    q, kv = d["q"].to(cuda), d["kv_cache"].to(cuda)
    out = torch.empty_like(q)
    lse = torch.empty((6, 32), dtype=torch.float32, device=cuda)
    _graph_equal(lambda: bskv.bskv_run_decode(p, q, kv, out=out, lse=lse), [out, lse])


def test_graph_bsr_tensor_cores_and_paged_prefill(cuda):
    d = synth.bsr_inputs(931, 512, 512, 64, 64, 8, 2, 128, pattern="diag_lower", causal=True)
    p = bskv.bskv_plan_bsr(d["indptr"], d["indices"], 512, 512, 64, 64, 8, 2, 128, causal=True)
    p.upload(cuda)
    q, k, v = d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda)
    out = torch.empty_like(q)
    f = synth.paged_prefill_inputs(932, 3, 8, 2, 128, 16, 0, 0, 0, 0, lengths=[300, 77, 129],
                                   qo_lens=[100, 77, 1])
    pp = bskv.bskv_plan_prefill_paged(f["qo_indptr"], f["kv_indptr"], f["kv_indices"],
                                      f["kv_last_page_len"], f["num_pages"], 16, 8, 2, 128)
    pp.upload(cuda)
    assert pp.metadata()[15] == 5
    fq, fkv = f["q"].to(cuda), f["kv_cache"].to(cuda)
    fout = torch.empty_like(fq)

    def run():
        bskv.bskv_run_bsr(p, q, k, v, out=out)
        bskv.bskv_run_prefill_paged(pp, fq, fkv, out=fout)

    _graph_equal(run, [out, fout])


def test_graph_mla_sparse(cuda):
    m = synth.mla_inputs(933, batch=2, heads=128, top_k=2048, pool_rows=4096, ctx_lo=2048,
                         ctx_hi=4096, max_seq_len=4096)
    g = {k: (v.to(cuda) if torch.is_tensor(v) else v) for k, v in m.items()}
    query = torch.empty((2, 1, 128, 576), dtype=torch.uint8, device=cuda)
    pool = torch.empty((4096, 576), dtype=torch.uint8, device=cuda)
    bskv.bskv_rope_quantize_fp8(g["q_rope"], g["k_rope"], g["q_nope"], g["k_nope"], g["cos_sin"],
                                g["pos_q"], True, q_rope_out=query[:, 0, :, 512:],
                                k_rope_out=pool[:, 512:], q_nope_out=query[:, 0, :, :512],
                                k_nope_out=pool[:, :512], pos_ids_k=g["pos_k"])
    p = bskv.bskv_plan_mla_sparse([2048, 2000], 2, 1, 128, 2048)
    p.upload(cuda)
    assert p.metadata()[5] > 0  # split pieces: the merge kernel is in the graph too
    out = torch.empty((2, 1, 128, 512), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((2, 1, 128), dtype=torch.float32, device=cuda)
    idx = g["indices"]
    _graph_equal(lambda: bskv.bskv_run_mla_sparse(p, query, pool, idx, 1 / math.sqrt(576), 1.0,
                                                  out=out, lse=lse), [out, lse])


def test_graph_mla_paged(cuda):
    """Dense paged MLA in a graph: whole tiles by TMA boxes of page slots, partial tiles
    gathered by rows, and (one long request) split pieces merged by the merge kernel."""
    d = synth.mla_paged_inputs(934, batch=3, heads=128, page_size=64, len_lo=0, len_hi=0,
                               lens=[2048, 300, 129])
    p = bskv.bskv_plan_mla_paged(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"], 3,
                                 d["num_pages"], 64, 128)
    p.upload(cuda)
    assert p.metadata()[6] > 0  # split pieces: the merge kernel is in the graph too
    q, kv = d["query"].to(cuda), d["kv_pages"].to(cuda)
    out = torch.empty((3, 128, 512), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((3, 128), dtype=torch.float32, device=cuda)
    _graph_equal(lambda: bskv.bskv_run_mla_paged(p, q, kv, 1 / math.sqrt(576), 1.0, out=out,
                                                 lse=lse), [out, lse])
