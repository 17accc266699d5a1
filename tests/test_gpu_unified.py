"""GPU parity for unified K/V blocks (JuliaPagedAttn README, "Features": the keys and values of a
token share one block, one block table and one pool).  Every call must give, on a unified pool
[num_blocks][2][block_size][n_kv_heads][head_dim], the same bits as on separate K and V pools
holding the same data, and match the oracle.  The layout travels with each call (the pools' block
stride), so calls on both layouts may run at the same time from different threads."""
import threading

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
    cuda_lib.set_checked_mode(False)
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
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    pa.paged_kv_write(k_new, v_new, slots, uk, uv)
    pa.copy_blocks(uk, uv, pairs)
    torch.cuda.synchronize()
    assert torch.equal(bits(u[:, 0]), bits(dk)) and torch.equal(bits(u[:, 1]), bits(dv))
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("D,G,S", [(128, 4, 16), (64, 1, 16), (128, 8, 32), (64, 2, 8), (128, 16, 16)])
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("split", [64, "none"])
def test_decode_unified_equals_separate(cuda_lib, dtype, D, G, S, kernel, split):
    pa = cuda_lib
    opts = dict(decode_kernel=kernel, partition_tokens=0 if split == "none" else split)
    ws = None if split == "none" else "auto"
    case = _decode_case(dtype, 2 * G, 2, D, S, [0, 1, S - 1, S, 100, 777], seed=D + G + S)
    q, k_new, v_new, slots, table, lens = _dev(case, "q", "k_new", "v_new", "slot_mapping", "block_table",
                                               "context_lens")
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    ref = pa.paged_attention_decode_fused(q, k_new, v_new, slots, dk, dv, table, lens, case.scale, workspace=ws,
                                          **opts)
    ref2 = pa.paged_attention_decode(q, dk, dv, table, lens, case.scale, workspace=ws, **opts)
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    out = pa.paged_attention_decode_fused(q, k_new, v_new, slots, uk, uv, table, lens, case.scale, workspace=ws,
                                          **opts)
    out2 = pa.paged_attention_decode(q, uk, uv, table, lens, case.scale, workspace=ws, **opts)
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(ref)) and torch.equal(bits(out2), bits(ref2))
    assert torch.equal(bits(u[:, 0]), bits(dk)) and torch.equal(bits(u[:, 1]), bits(dv))
    assert pa.device_error_flags() == 0


def test_decode_unified_matches_the_oracle_on_the_serving_batch(cuda_lib):
    pa = cuda_lib
    case = W.llama_decode()
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
@pytest.mark.parametrize("kernel", [1, 2])
def test_prefill_unified_equals_separate(cuda_lib, dtype, kernel):
    """kernel 1 = CUDA cores, 2 = tcgen05; mixed decode rows and prefill chunks."""
    pa = cuda_lib
    case = W.varlen_prefill(123, hist_lens=[700, 0, 95, 33, 260], chunk_lens=[1, 128, 1, 64, 200], block_size=16,
                            n_q_heads=32, n_kv_heads=8, head_dim=128, dtype=dtype, num_blocks=160)
    q, qsl, table, lens, k_new, v_new, slots = _dev(case, "q", "query_start_loc", "block_table", "context_lens",
                                                    "k_new", "v_new", "slot_mapping")
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(k_new, v_new, slots, dk, dv)
    ref = pa.paged_attention_prefill(q, qsl, dk, dv, table, lens, case.scale, prefill_kernel=kernel)
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    pa.paged_kv_write(k_new, v_new, slots, uk, uv)
    out = pa.paged_attention_prefill(q, qsl, uk, uv, table, lens, case.scale, prefill_kernel=kernel)
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


def test_mismatched_layouts_are_refused(cuda_lib):
    pa = cuda_lib
    case = _decode_case(torch.bfloat16, 8, 2, 128, 16, [40, 90], seed=5)
    q, table, lens = _dev(case, "q", "block_table", "context_lens")
    dk = case.k_pool.cuda()
    u = unify(case.k_pool, case.v_pool).cuda()
    uk, uv = pa.unified_views(u)
    with pytest.raises(ValueError):  # K contiguous, V a view of a unified pool: two block strides
        pa.paged_attention_decode(q, dk, uv, table, lens, case.scale)
    host = torch.empty((8,) + tuple(u.shape[1:]), dtype=u.dtype).pin_memory()
    hk = torch.empty((8,) + tuple(case.k_pool.shape[1:]), dtype=u.dtype).pin_memory()
    pairs = torch.tensor([[0, 1]], dtype=torch.int64).cuda()
    with pytest.raises(ValueError):  # unified device pool into separate host pools
        pa.swap_blocks(hk, hk.clone().pin_memory(), uk, uv, pairs)
    del host
    # the C ABI: a block stride that is not a multiple of 16 bytes, or shorter than one block
    lib = pa.load_library()
    out = torch.empty_like(q)
    for stride in (2 * 16 * 2 * 128 * 2 + 8, 16 * 2 * 128 * 2 - 16):
        o = pa.make_opts(kv_block_stride_bytes=stride)
        import ctypes
        st = lib.paged_attention_decode_ex(out.data_ptr(), q.data_ptr(), uk.data_ptr(), uv.data_ptr(),
                                           table.data_ptr(), int(table.shape[1]), lens.data_ptr(), int(q.shape[0]),
                                           int(u.shape[0]), 16, case.scale, 8, 2, 128, pa.PA_BF16, None, 0,
                                           ctypes.byref(o), None)
        assert st == pa.PA_EINVAL


def test_both_layouts_from_two_threads_at_once(cuda_lib):
    """One thread decodes and prefills on separate pools while another does the same on a unified
    pool, each on its own stream, many calls interleaved: both match the oracle (the layout is a
    per-call argument, so neither thread can change what the other computes)."""
    pa = cuda_lib
    case = _decode_case(torch.bfloat16, 32, 8, 128, 16, [300, 1500, 40, 777, 2100], seed=61)
    pc = W.varlen_prefill(62, hist_lens=[500, 0, 95], chunk_lens=[64, 128, 1], block_size=16, n_q_heads=32,
                          n_kv_heads=8, head_dim=128, dtype=torch.bfloat16, num_blocks=64)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref_dec = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    pk1, pv1 = oracle.paged_kv_write(pc.k_pool, pc.v_pool, pc.k_new, pc.v_new, pc.slot_mapping)
    ref_pf = oracle.paged_prefill(pc.q, pc.query_start_loc, pk1, pv1, pc.block_table, pc.context_lens, pc.scale)
    idx = sorted(ref_pf)
    ref_pf = np.stack([ref_pf[i] for i in idx])
    results, errors = {}, []

    def worker(layout):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                q, k_new, v_new, slots, table, lens = _dev(case, "q", "k_new", "v_new", "slot_mapping",
                                                           "block_table", "context_lens")
                pq, qsl, ptable, plens, pkn, pvn, pslots = _dev(pc, "q", "query_start_loc", "block_table",
                                                                "context_lens", "k_new", "v_new", "slot_mapping")
                if layout == "unified":
                    u, pu = unify(case.k_pool, case.v_pool).cuda(), unify(pc.k_pool, pc.v_pool).cuda()
                    kp, vp = pa.unified_views(u)
                    pkp, pvp = pa.unified_views(pu)
                else:
                    kp, vp = case.k_pool.cuda(), case.v_pool.cuda()
                    pkp, pvp = pc.k_pool.cuda(), pc.v_pool.cuda()
                pa.paged_kv_write(k_new, v_new, slots, kp, vp, stream=stream)
                pa.paged_kv_write(pkn, pvn, pslots, pkp, pvp, stream=stream)
                outs = []
                for i in range(20):
                    d = pa.paged_attention_decode(q, kp, vp, table, lens, case.scale, stream=stream,
                                                  partition_tokens=256 if i % 2 else 0)
                    p = pa.paged_attention_prefill(pq, qsl, pkp, pvp, ptable, plens, pc.scale, stream=stream)
                    outs.append((d, p))
                stream.synchronize()
                results[layout] = [(d.cpu(), p.cpu()) for d, p in outs]
        except Exception as e:  # surfaced by the main thread
            errors.append((layout, repr(e)))

    threads = [threading.Thread(target=worker, args=(lay,)) for lay in ("separate", "unified")]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for layout in ("separate", "unified"):
        for d, p in results[layout]:
            assert np.abs(d.double().numpy() - ref_dec).max() <= 2e-2, layout
            assert np.abs(p[idx].double().numpy() - ref_pf).max() <= 2e-2, layout
    assert pa.device_error_flags() == 0
