"""The no-allocation decode entry point, paged_attention_decode_static_scratch.

It serves callers that cannot allocate device memory (a plugin host that owns the allocator, a
serving loop whose memory plan is fixed at start-up, a caller holding only raw pointers): it
takes its split-K scratch from a fixed device array inside the library instead of a caller
workspace.  Here it is called through the C ABI and compared with paged_attention_decode (which
uses a caller workspace) on two calls in a row, so that contents the first call leaves in the
shared array cannot leak into the second.  This file is collected last on purpose.
"""
import ctypes
import math

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _call_static(lib, out, case, q, lens, table):
    st = lib.paged_attention_decode_static_scratch(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(case["kp"].data_ptr()),
        ctypes.c_void_p(case["vp"].data_ptr()), ctypes.c_void_p(table.data_ptr()), table.stride(0),
        ctypes.c_void_p(lens.data_ptr()), q.shape[0], case["kp"].shape[0], case["kp"].shape[1],
        1.0 / math.sqrt(q.shape[2]), q.shape[1], case["kp"].shape[2], q.shape[2], 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_static_scratch_decode_matches_workspace_decode_twice(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    # 256-token partitions: 512..4096-token contexts split into up to 16 partitions, more than one
    # thread-block cluster holds, so the partial states go through the scratch array and the merge
    pa.set_option(pa.PA_OPT_PARTITION_TOKENS, 256)
    lens = W.llama_context_lens()
    inp = W.device_decode_inputs(lens, n_q_heads=32, n_kv_heads=8, head_dim=128, block_size=16,
                                 dtype=torch.bfloat16, num_blocks=W.LLAMA_POOL,
                                 max_blocks_per_seq=W.LLAMA_MAX_CTX // 16, device="cuda", seed=2024)
    kp, vp = inp["pools"][0]
    case = {"kp": kp, "vp": vp}
    table = inp["block_table"].cuda()
    need = pa.decode_workspace_size(64, table.stride(0), 16, 32, 8, 128)
    assert 0 < need <= pa.PA_STATIC_SCRATCH_BYTES
    gen = torch.Generator().manual_seed(77)
    for call in range(2):
        q = (torch.randn((64, 32, 128), generator=gen) * (1 + 3 * call)).to(torch.bfloat16).cuda()
        # the second call shortens every context so stale partitions of the first would be wrong
        ctx = inp["context_lens"].cuda() - 300 * call
        ref = pa.paged_attention_decode(q, kp, vp, table, ctx)
        out = torch.full_like(q, float("nan"))
        assert _call_static(lib, out, case, q, ctx, table) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= 2e-2, f"call {call}: max abs err {err}"
    assert pa.device_error_flags() == 0
    pa.set_option(pa.PA_OPT_PARTITION_TOKENS, 0)


def test_static_scratch_rejects_problems_larger_than_the_array(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    # 4 x 131072-token tables with 512-token partitions need ~17 MB; 64 such rows need far more
    n = 64
    stride = 131072 // 16
    need = pa.decode_workspace_size(n, stride, 16, 32, 8, 128)
    assert need > pa.PA_STATIC_SCRATCH_BYTES
    null = ctypes.c_void_p(0)
    st = lib.paged_attention_decode_static_scratch(null, null, null, null, null, stride, null, n, 1000, 16,
                                                   0.1, 32, 8, 128, 0, null)
    assert st == pa.PA_EWORKSPACE
