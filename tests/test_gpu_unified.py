"""GPU parity for unified K/V blocks (JuliaPagedAttn README, "Features": the keys and values of a
token share one block, one block table and one pool).  Every call must give, on a unified pool
[num_blocks][2][block_size][n_kv_heads][head_dim], the same bits as on separate K and V pools
holding the same data, and match the oracle; the library must refuse pools whose layout does not
match the selected one."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int16) if t.element_size() == 2 else t.contiguous().view(torch.int32)


def unify(k_pool, v_pool):
    """Unified pool holding the blocks of separate pools: block b = (K block b, V block b)."""
    return torch.stack([k_pool, v_pool], dim=1).contiguous()


@pytest.fixture(autouse=True)
def _reset(cuda_lib):
    yield
    for opt in (cuda_lib.PA_OPT_KV_LAYOUT, cuda_lib.PA_OPT_DECODE_KERNEL, cuda_lib.PA_OPT_PARTITION_TOKENS,
                cuda_lib.PA_OPT_PREFILL_KERNEL, cuda_lib.PA_OPT_CHECKED, cuda_lib.PA_OPT_CLUSTER_MERGE):
        cuda_lib.set_option(opt, 0)
    cuda_lib.device_error_flags(clear=True)


def _decode_case(dtype, Hq, Hkv, D, S, lens, seed):
    need = sum(W.ceil_div(n + 1, S) for n in lens)
    maxb = max(W.ceil_div(n + 1, S) for n in lens) + 1
    return W.decode_case(f"unified_{seed}", seed, lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, block_size=S,
                         dtype=dtype, num_blocks=need + 7, max_blocks_per_seq=maxb)


def _dev(case, *names):
    return [getattr(case, n).cuda() for n in names]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_kv_write_and_copy_blocks_on_a_unified_pool(cuda_lib, dtype):
    pa = cuda_lib
    case = _decode_case(dtype, 8, 2, 128, 16, [0, 5, 16, 40, 333], seed=11)
    k_new, v_new, slots = _dev(case, "k_new", "v_new", "slot_mapping")
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(k_new, v_new, slots, dk, dv)
    pairs = torch.tensor([[case.block_table[3, 0].item(), case.k_pool.shape[0] - 1],
                          [case.block_table[4, 2].item(), case.k_pool.shape[0] - 2]], dtype=torch.int64).cuda()
    pa.copy_blocks(dk, dv, pairs)
    pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    pa.paged_kv_write(k_new, v_new, slots, uk, uv)
    pa.copy_blocks(uk, uv, pairs)
    torch.cuda.synchronize()
    assert torch.equal(bits(u[:, 0]), bits(dk)) and torch.equal(bits(u[:, 1]), bits(dv))
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("D,G,S", [(128, 4, 16), (64, 1, 16), (128, 8, 32), (64, 2, 8)])
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("split", [64, "none", "cluster"])
def test_decode_unified_equals_separate(cuda_lib, dtype, D, G, S, kernel, split):
    pa = cuda_lib
    pa.set_option(pa.PA_OPT_DECODE_KERNEL, kernel)
    if split == "cluster":
        pa.set_option(pa.PA_OPT_CLUSTER_MERGE, 1)
        pa.set_option(pa.PA_OPT_PARTITION_TOKENS, 128)
    elif split != "none":
        pa.set_option(pa.PA_OPT_PARTITION_TOKENS, split)
    ws = None if split == "none" else "auto"
    case = _decode_case(dtype, 2 * G, 2, D, S, [0, 1, S - 1, S, 100, 777], seed=D + G + S)
    q, k_new, v_new, slots, table, lens = _dev(case, "q", "k_new", "v_new", "slot_mapping", "block_table",
                                               "context_lens")
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    ref = pa.paged_attention_decode_fused(q, k_new, v_new, slots, dk, dv, table, lens, case.scale, workspace=ws)
    ref2 = pa.paged_attention_decode(q, dk, dv, table, lens, case.scale, workspace=ws)
    pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    out = pa.paged_attention_decode_fused(q, k_new, v_new, slots, uk, uv, table, lens, case.scale, workspace=ws)
    out2 = pa.paged_attention_decode(q, uk, uv, table, lens, case.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(ref)) and torch.equal(bits(out2), bits(ref2))
    assert torch.equal(bits(u[:, 0]), bits(dk)) and torch.equal(bits(u[:, 1]), bits(dv))
    assert pa.device_error_flags() == 0


def test_decode_unified_matches_the_oracle_on_the_serving_batch(cuda_lib):
    pa = cuda_lib
    case = W.llama_decode()
    pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    q, k_new, v_new, slots, table, lens = _dev(case, "q", "k_new", "v_new", "slot_mapping", "block_table",
                                               "context_lens")
    out = pa.paged_attention_decode_fused(q, k_new, v_new, slots, uk, uv, table, lens, case.scale).cpu()
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    rows = [(b, h) for b in range(1, 64, 5) for h in (2, 7)]
    ref = oracle.paged_decode_rows(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale, rows)
    for (b, h), r in ref.items():
        err = np.abs(out[b, 4 * h:4 * h + 4].double().numpy() - r).max()
        assert err <= 2e-2, (b, h, err)
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_prefill_unified_equals_separate(cuda_lib, dtype, kernel):
    """kernel 1 = CUDA cores, 2 = tcgen05, 3 = mma.sync; mixed decode rows and prefill chunks."""
    pa = cuda_lib
    pa.set_option(pa.PA_OPT_PREFILL_KERNEL, kernel)
    case = W.varlen_prefill(123, hist_lens=[700, 0, 95, 33, 260], chunk_lens=[1, 128, 1, 64, 200], block_size=16,
                            n_q_heads=32, n_kv_heads=8, head_dim=128, dtype=dtype, num_blocks=160)
    q, qsl, table, lens, k_new, v_new, slots = _dev(case, "q", "query_start_loc", "block_table", "context_lens",
                                                    "k_new", "v_new", "slot_mapping")
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(k_new, v_new, slots, dk, dv)
    ref = pa.paged_attention_prefill(q, qsl, dk, dv, table, lens, case.scale)
    pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    pa.paged_kv_write(k_new, v_new, slots, uk, uv)
    out = pa.paged_attention_prefill(q, qsl, uk, uv, table, lens, case.scale)
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(ref))
    kp, vp = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens, case.scale)
    idx = sorted(res)
    err = np.abs(out.cpu()[idx].double().numpy() - np.stack([res[i] for i in idx])).max()
    assert err <= 2e-2
    assert pa.device_error_flags() == 0


def test_swap_unified_pools_round_trip(cuda_lib):
    pa = cuda_lib
    case = _decode_case(torch.bfloat16, 8, 2, 128, 16, [40, 333, 90], seed=21)
    pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
    u = unify(case.k_pool, case.v_pool).cuda()
    host = torch.empty((8,) + tuple(u.shape[1:]), dtype=u.dtype).pin_memory()
    blocks = [int(x) for x in case.block_table[1, :8]]
    out_pairs = torch.tensor([[b, i] for i, b in enumerate(blocks)], dtype=torch.int64).pin_memory()
    pa.swap_blocks(*pa.unified_views(host), *pa.unified_views(u), out_pairs)
    torch.cuda.synchronize()
    assert torch.equal(bits(host), bits(u[blocks].cpu()))
    free = [case.k_pool.shape[0] - 1 - i for i in range(8)]
    in_pairs = torch.tensor([[i, f] for i, f in enumerate(free)], dtype=torch.int64).cuda()
    pa.swap_blocks(*pa.unified_views(u), *pa.unified_views(host), in_pairs)
    torch.cuda.synchronize()
    assert torch.equal(bits(u[free].cpu()), bits(host))
    assert pa.device_error_flags() == 0


def test_layout_mismatch_is_refused(cuda_lib):
    pa = cuda_lib
    case = _decode_case(torch.bfloat16, 8, 2, 128, 16, [40, 90], seed=5)
    q, table, lens = _dev(case, "q", "block_table", "context_lens")
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    with pytest.raises(ValueError):  # unified views while the separate layout is selected
        pa.paged_attention_decode(q, uk, uv, table, lens, case.scale)
    pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
    with pytest.raises(ValueError):  # separate pools while the unified layout is selected
        pa.paged_attention_decode(q, dk, dv, table, lens, case.scale)
    # the C ABI itself: v_pool must be the V half of block 0
    lib = pa.load_library()
    out = torch.empty_like(q)
    st = lib.paged_attention_decode(out.data_ptr(), q.data_ptr(), uk.data_ptr(), uk.data_ptr() + 16, table.data_ptr(),
                                    int(table.shape[1]), lens.data_ptr(), int(q.shape[0]), int(u.shape[0]), 16,
                                    case.scale, 8, 2, 128, pa.PA_BF16, None, 0, None)
    assert st == pa.PA_EINVAL
    swapped = torch.stack([case.v_pool, case.k_pool], dim=1).contiguous().cuda()  # V first: not a unified pool
    st = lib.copy_blocks(swapped[:, 1].data_ptr(), swapped[:, 0].data_ptr(), None, 0, int(u.shape[0]),
                         16 * 2 * 128 * 2, None)
    assert st == pa.PA_OK  # n_pairs == 0 is a no-op before any check
    pairs = torch.tensor([[0, 1]], dtype=torch.int64).cuda()
    st = lib.copy_blocks(swapped[:, 1].data_ptr(), swapped[:, 0].data_ptr(), pairs.data_ptr(), 1, int(u.shape[0]),
                         16 * 2 * 128 * 2, None)
    assert st == pa.PA_EINVAL
