"""GPU parity for swap_blocks: moving blocks between the device pool and a pinned host pool
(Pico-vLLM dev log #5 "Paged Attention": swap_out / swap_in), bit-exact against the oracle, and a
swap-out / swap-in round trip that leaves decode attention unchanged."""
import ctypes

import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.fixture(autouse=True)
def _reset(cuda_lib):
    yield
    cuda_lib.set_checked_mode(False)
    cuda_lib.device_error_flags(clear=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("where", ["out", "in", "device"])
def test_swap_bit_exact(cuda_lib, dtype, where):
    pa = cuda_lib
    gen = torch.Generator().manual_seed(31)
    dev_k = W.randn(gen, (60, 16, 8, 128), dtype)
    dev_v = W.randn(gen, (60, 16, 8, 128), dtype)
    host_k = W.randn(gen, (40, 16, 8, 128), dtype)
    host_v = W.randn(gen, (40, 16, 8, 128), dtype)
    pairs = torch.tensor([[3, 0], [17, 39], [59 if where != "in" else 39, 5], [0, 1]], dtype=torch.int64)
    if where == "out":      # device -> pinned host
        src, dst = (dev_k, dev_v), (host_k, host_v)
        s_dev = (src[0].cuda(), src[1].cuda())
        d_dev = (dst[0].pin_memory(), dst[1].pin_memory())
        p = pairs.cuda()
    elif where == "in":     # pinned host -> device
        src, dst = (host_k, host_v), (dev_k, dev_v)
        s_dev = (src[0].pin_memory(), src[1].pin_memory())
        d_dev = (dst[0].cuda(), dst[1].cuda())
        p = pairs.pin_memory()
    else:                   # device -> another device pool
        src, dst = (dev_k, dev_v), (dev_k.clone(), dev_v.clone())
        s_dev = (src[0].cuda(), src[1].cuda())
        d_dev = (dst[0].cuda(), dst[1].cuda())
        p = pairs.cuda()
    pa.swap_blocks(d_dev[0], d_dev[1], s_dev[0], s_dev[1], p)
    torch.cuda.synchronize()
    ref_k, ref_v = oracle.transfer_blocks(dst[0], dst[1], src[0], src[1], pairs)
    assert torch.equal(bits(d_dev[0].cpu()), bits(ref_k)) and torch.equal(bits(d_dev[1].cpu()), bits(ref_v))
    assert pa.device_error_flags() == 0


def test_swap_out_and_back_leaves_attention_unchanged(cuda_lib):
    """Swap a sequence's blocks to the host pool, bring them back into different physical blocks,
    retarget the table: decode attention gives the same bits (the reduction depends only on logical
    positions)."""
    pa = cuda_lib
    case = W.decode_case("swap_rt", 77, [300, 170, 513], n_q_heads=32, n_kv_heads=8, head_dim=128, block_size=16,
                         dtype=torch.bfloat16, num_blocks=120, max_blocks_per_seq=40)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    table = case.block_table.cuda()
    lens = case.context_lens.cuda()
    before = pa.paged_attention_decode(case.q.cuda(), dk, dv, table, lens, case.scale).cpu()
    used = case.block_table[0][case.block_table[0] >= 0]
    n = used.numel()
    host_k = torch.zeros((n, 16, 8, 128), dtype=torch.bfloat16).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_pairs = torch.stack([used.to(torch.int64), torch.arange(n, dtype=torch.int64)], dim=1)
    pa.swap_blocks(host_k, host_v, dk, dv, out_pairs.cuda())
    # free the device blocks (overwrite them) and bring the data back into fresh blocks
    all_used = set(int(x) for x in case.block_table.flatten() if x >= 0)
    fresh = [b for b in range(case.num_blocks) if b not in all_used][:n]
    dk[used.cuda().long()] = 0
    dv[used.cuda().long()] = 0
    in_pairs = torch.stack([torch.arange(n, dtype=torch.int64), torch.tensor(fresh, dtype=torch.int64)], dim=1)
    pa.swap_blocks(dk, dv, host_k, host_v, in_pairs.pin_memory())
    new_table = case.block_table.clone()
    new_table[0, :n] = torch.tensor(fresh, dtype=torch.int32)
    after = pa.paged_attention_decode(case.q.cuda(), dk, dv, new_table.cuda(), lens, case.scale).cpu()
    assert torch.equal(bits(before), bits(after))
    assert pa.device_error_flags() == 0


def test_swap_errors(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    k = torch.zeros((4, 16, 2, 64), dtype=torch.float16, device="cuda")
    v = torch.zeros_like(k)
    hk = torch.ones((4, 16, 2, 64), dtype=torch.float16).pin_memory()
    hv = torch.ones_like(hk).pin_memory()
    pa.swap_blocks(k, v, hk, hv, torch.tensor([[1, 2], [0, 7]], dtype=torch.int64, device="cuda"))
    assert pa.device_error_flags() & pa.PA_DEVERR_COPY_PAIR
    assert float(k[2].float().min()) == 1.0
    # pageable host memory cannot be reached from the device: rejected before any launch
    pageable = torch.ones((4, 16, 2, 64), dtype=torch.float16)
    st = lib.swap_blocks(ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()), 4,
                         ctypes.c_void_p(pageable.data_ptr()), ctypes.c_void_p(pageable.data_ptr()), 4,
                         ctypes.c_void_p(torch.zeros((1, 2), dtype=torch.int64, device="cuda").data_ptr()), 1,
                         16 * 2 * 64 * 2, None)
    assert st == pa.PA_EINVAL
    pa.set_checked_mode(True)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.swap_blocks(k, v, hk, hv, torch.tensor([[1, 2], [3, 2]], dtype=torch.int64, device="cuda"))
    assert ei.value.status == pa.PA_ERANGE
