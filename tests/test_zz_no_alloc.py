"""The no-allocation decode entry point, paged_attention_decode_static_scratch.

It serves callers that cannot allocate device memory (a plugin host that owns the allocator, a
serving loop whose memory plan is fixed at start-up, a caller holding only raw pointers): it
takes its split-K scratch from a fixed device array inside the library instead of a caller
workspace.  Here it is called through the C ABI and compared with paged_attention_decode (which
uses a caller workspace) on two calls in a row, so that contents the first call leaves in the
shared array cannot leak into the second.  Both take the same split-K plan and the same kernels,
so the outputs must be bit-identical; sampled rows are also checked against the CPU oracle.  This
file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def _call_static(lib, out, kp, vp, q, lens, table, stream=None):
    return lib.paged_attention_decode_static_scratch(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), ctypes.c_void_p(table.data_ptr()), table.stride(0),
        ctypes.c_void_p(lens.data_ptr()), q.shape[0], kp.shape[0], kp.shape[1],
        1.0 / math.sqrt(q.shape[2]), q.shape[1], kp.shape[2], q.shape[2], 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream if stream is None else stream))


def test_static_scratch_decode_matches_workspace_decode_twice(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    # the serving batch: 512..4096-token contexts split into up to 4 partitions of 1024 tokens, so
    # the partial states go through the scratch array and the merge kernel
    case = W.llama_decode()
    kp, vp = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), kp, vp)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    table = case.block_table.cuda()
    need = pa.decode_workspace_size(64, table.stride(0), 16, 32, 8, 128)
    assert 0 < need <= pa.PA_STATIC_SCRATCH_BYTES
    gen = torch.Generator().manual_seed(77)
    for call in range(2):
        q = (torch.randn((64, 32, 128), generator=gen) * (1 + 3 * call)).to(torch.bfloat16)
        # the second call shortens every context so stale partitions of the first would be wrong
        lens = case.context_lens - 300 * call
        ref = pa.paged_attention_decode(q.cuda(), kp, vp, table, lens.cuda(), 1.0 / math.sqrt(128))
        out = torch.full((64, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_static(lib, out, kp, vp, q.cuda(), lens.cuda(), table) == 0
        torch.cuda.synchronize()
        got = out.cpu()
        assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16)), f"call {call}: bits differ"
        rows = [(b, h) for b in range(call, 64, 9) for h in (1, 6)]
        want = oracle.paged_decode_rows(q, kp1, vp1, case.block_table, lens, 1.0 / math.sqrt(128), rows)
        for (b, h), r in want.items():
            err = np.abs(got[b, 4 * h:4 * h + 4].double().numpy() - r).max()
            assert err <= 2e-2, (call, b, h, err)
    assert pa.device_error_flags() == 0


def test_static_scratch_rejects_problems_larger_than_the_array(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    # 64 rows of 131072-token tables split into 128 partitions of 1024 tokens: 136 MB of scratch
    n, stride = 64, 131072 // 16
    need = pa.decode_workspace_size(n, stride, 16, 32, 8, 128)
    assert need > pa.PA_STATIC_SCRATCH_BYTES
    q = torch.zeros((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    kp = torch.zeros((16, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    table = torch.zeros((n, stride), dtype=torch.int32, device="cuda")
    lens = torch.full((n,), 131072, dtype=torch.int32, device="cuda")
    before = pa.launch_count()
    assert _call_static(lib, out, kp, vp, q, lens, table) == pa.PA_EWORKSPACE
    assert pa.launch_count() == before  # rejected before anything was launched
    # arguments are checked before the size: a bad dtype or group is reported as such
    st = lib.paged_attention_decode_static_scratch(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), ctypes.c_void_p(table.data_ptr()), stride, ctypes.c_void_p(lens.data_ptr()),
        n, 16, 16, 0.1, 32, 8, 128, 9, None)
    assert st == pa.PA_EDTYPE
    st = lib.paged_attention_decode_static_scratch(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), ctypes.c_void_p(table.data_ptr()), stride, ctypes.c_void_p(lens.data_ptr()),
        n, 16, 16, 0.1, 32, 1, 128, 0, None)
    assert st == pa.PA_EUNSUPPORTED  # 32 query heads per KV head
