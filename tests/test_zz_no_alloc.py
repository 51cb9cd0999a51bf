"""The allocation-free paged decode entry point, checked against the regular one.

bskv_run_decode_noalloc serves callers that cannot allocate device memory (code that is
handed only tensors and a stream by its host framework, processes whose device memory is
reserved by another allocator, loops where cudaMalloc's device synchronisation is not
acceptable). It keeps the plan metadata and the split-KV partial states in static device
arrays owned by the library. This file calls it through the C ABI twice in a row, on two
different workloads and plans (both cut some requests into split-KV pieces, so the
static scratch holds partial states; the test asserts that before the call), and compares
each result with bskv_run_decode's bit for bit: both run the same attention kernel and the
same log-sum-exp merge in the same order, only the memory that holds the metadata and the
partial states differs. It also checks that a plan too large for the static arrays is
refused before anything is launched. The file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth

pytestmark = pytest.mark.gpu
H_MERGES = 6  # metadata header word: number of split units the merge combines


def _strides(*v):
    return (ctypes.c_int64 * len(v))(*v)


def _noalloc(lib, plan, q, kv, out, lse, scale):
    ks = kv.stride()
    return lib.bskv_run_decode_noalloc(
        plan.handle, q.data_ptr(), _strides(q.stride(0), q.stride(1)), kv.data_ptr(),
        _strides(ks[0], ks[1], ks[2], ks[3]), out.data_ptr(),
        _strides(out.stride(0), out.stride(1)), lse.data_ptr(), ctypes.c_float(scale),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_regular_entry_twice(cuda):
    lib = bskv.load_library()
    for seed, max_workers in [(910, 0), (911, 37)]:
        d = synth.paged_decode_inputs(seed, 6, 32, 8, 128, 16, 1, 2000)
        plan = bskv.bskv_plan_decode(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"],
                                     d["num_pages"], 16, 32, 8, 128, torch.bfloat16,
                                     max_workers=max_workers)
        # the plan splits some requests, so the call goes through the static scratch array
        assert plan.workspace_sizes()[1] > 0 and plan.metadata()[H_MERGES] > 0
        q, kv = d["q"].to(cuda), d["kv_cache"].to(cuda)
        ref, ref_lse = bskv.bskv_run_decode(plan, q, kv, return_lse=True)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((6, 32), float("nan"), dtype=torch.float32, device=cuda)
        code = _noalloc(lib, plan, q, kv, out, lse, d["sm_scale"])
        assert code == 0, bskv.bskv_last_error_message()
        torch.cuda.synchronize()
        assert bskv.bskv_get_device_status() == 0
        assert torch.equal(out, ref), "out (seed %d)" % seed
        assert torch.equal(lse, ref_lse), "lse (seed %d)" % seed


def test_noalloc_rejects_a_plan_beyond_the_static_arrays(cuda):
    lib = bskv.load_library()
    # one long request, 16 query heads per kv head, many workers: > 8 MiB of partials
    indptr = torch.tensor([0, 4000], dtype=torch.int32)
    idx = torch.arange(4000, dtype=torch.int32)
    last = torch.tensor([16], dtype=torch.int32)
    plan = bskv.bskv_plan_decode(indptr, idx, last, 4000, 16, 16, 1, 128, torch.bfloat16,
                                 max_workers=2000)
    assert plan.workspace_sizes()[1] > (8 << 20)
    t = torch.zeros((1, 16, 128), dtype=torch.bfloat16, device=cuda)
    lse = torch.zeros((1, 16), dtype=torch.float32, device=cuda)
    kv = torch.zeros((1, 2, 1, 16, 128), dtype=torch.bfloat16, device=cuda)
    code = _noalloc(lib, plan, t, kv, t, lse, 0.1)
    assert bskv.STATUS[code] == "ERR_UNSUPPORTED"
    assert "static arrays hold" in bskv.bskv_last_error_message()
