"""Failure detection on the GPU without a fault: the bounded waits of the pipelined kernels.

Every TMA ring and tensor-memory hand-off waits on an mbarrier with a time limit; when the limit
runs out the kernel records PA_DEVERR_TIMEOUT and returns, and the other waiting warps leave as soon
as they see that bit.  pa_selftest_bounded_wait runs that path on barriers nothing completes (a flag
that nothing sets), so the test checks the status, the limits, that the context stays usable and that the abort stays
with the launch that gave up."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(cuda_lib):
    pa = cuda_lib
    pa.device_error_flags(clear=True)
    flags, w0, w1 = pa.selftest_bounded_wait(20_000_000)  # 20 ms
    assert flags == pa.PA_DEVERR_TIMEOUT
    assert 20_000_000 <= w0 < 500_000_000, w0
    # warp 1's own limit is 1 s; it left once warp 0 had raised the bit
    assert w1 < 500_000_000, w1
    assert pa.device_error_flags() == 0  # read and cleared above
    # the context still works: a decode call right after matches the oracle
    case = W.decode_case("after_timeout", 77, [40, 300], n_q_heads=8, n_kv_heads=2, head_dim=64, block_size=16,
                         dtype=torch.bfloat16, num_blocks=40, max_blocks_per_seq=24)
    lens = case.context_lens - 1
    out = pa.paged_attention_decode(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(), case.block_table.cuda(),
                                    lens.cuda(), case.scale).cpu()
    ref = oracle.paged_decode(case.q, case.k_pool, case.v_pool, case.block_table, lens, case.scale)
    assert abs(out.double().numpy() - ref).max() <= 2e-2
    assert pa.device_error_flags() == 0


def test_selftest_limits_are_checked(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    assert lib.pa_selftest_bounded_wait(10, None, None) == pa.PA_EINVAL
    assert lib.pa_selftest_bounded_wait(2_000_000_000, None, None) == pa.PA_EINVAL


def test_a_timeout_left_uncleared_does_not_cut_later_launches_short(cuda_lib):
    """The abort a timed-out wait publishes belongs to its own launch: with PA_DEVERR_TIMEOUT still
    set (not cleared), a later decode (pipelined TMA waits) and prefill (tcgen05 hand-offs) run to
    completion and match the oracle, and the bit stays reported until it is cleared."""
    pa = cuda_lib
    pa.device_error_flags(clear=True)
    flags, _, w1 = pa.selftest_bounded_wait(5_000_000, clear=False)  # 5 ms; the flags stay set
    assert flags == pa.PA_DEVERR_TIMEOUT and w1 < 500_000_000
    case = W.decode_case("after_uncleared_timeout", 78, [40, 300, 1500, 3000], n_q_heads=32, n_kv_heads=8,
                         head_dim=128, block_size=16, dtype=torch.bfloat16, num_blocks=320, max_blocks_per_seq=200)
    lens = case.context_lens - 1
    out = pa.paged_attention_decode(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(), case.block_table.cuda(),
                                    lens.cuda(), case.scale, partition_tokens=256).cpu()
    ref = oracle.paged_decode(case.q, case.k_pool, case.v_pool, case.block_table, lens, case.scale)
    assert abs(out.double().numpy() - ref).max() <= 2e-2
    pc = W.varlen_prefill(79, hist_lens=[300, 0, 129], chunk_lens=[200, 64, 17], block_size=16, n_q_heads=32,
                          n_kv_heads=8, head_dim=128, dtype=torch.bfloat16, num_blocks=64)
    pk, pv = pc.k_pool.cuda(), pc.v_pool.cuda()
    pa.paged_kv_write(pc.k_new.cuda(), pc.v_new.cuda(), pc.slot_mapping.cuda(), pk, pv)
    pout = pa.paged_attention_prefill(pc.q.cuda(), pc.query_start_loc.cuda(), pk, pv, pc.block_table.cuda(),
                                      pc.context_lens.cuda(), pc.scale).cpu()
    okp, ovp = oracle.paged_kv_write(pc.k_pool, pc.v_pool, pc.k_new, pc.v_new, pc.slot_mapping)
    res = oracle.paged_prefill(pc.q, pc.query_start_loc, okp, ovp, pc.block_table, pc.context_lens, pc.scale)
    idx = sorted(res)
    assert abs(pout[idx].double().numpy() - np.stack([res[i] for i in idx])).max() <= 2e-2
    assert pa.device_error_flags(clear=False) == pa.PA_DEVERR_TIMEOUT  # still reported
    assert pa.device_error_flags(clear=True) == pa.PA_DEVERR_TIMEOUT
    assert pa.device_error_flags() == 0
