"""GPU parity for the fused write + decode (nanoserve Day 19, "What I added today": write this step's
K/V to its slot, then attend over the whole history through the block table).  The fused call must
leave the same bits in the output and in both pools as paged_kv_write followed by
paged_attention_decode, and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float16, torch.float32]


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.fixture(autouse=True)
def _reset(cuda_lib):
    yield
    cuda_lib.set_checked_mode(False)
    cuda_lib.device_error_flags(clear=True)


def _case(dtype, Hq, Hkv, D, S, lens, seed):
    need = sum(W.ceil_div(n + 1, S) for n in lens)
    maxb = max(W.ceil_div(n + 1, S) for n in lens) + 1
    return W.decode_case(f"fused_{seed}", seed, lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, block_size=S,
                         dtype=dtype, num_blocks=need + 5, max_blocks_per_seq=maxb)


def _both(pa, case, workspace="auto", **opts):
    dev = {k: getattr(case, k).cuda() for k in ("q", "k_new", "v_new", "slot_mapping", "block_table", "context_lens")}
    k1, v1 = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], k1, v1)
    ref = pa.paged_attention_decode(dev["q"], k1, v1, dev["block_table"], dev["context_lens"], case.scale,
                                    workspace=workspace, **opts)
    k2, v2 = case.k_pool.cuda(), case.v_pool.cuda()
    out = pa.paged_attention_decode_fused(dev["q"], dev["k_new"], dev["v_new"], dev["slot_mapping"], k2, v2,
                                          dev["block_table"], dev["context_lens"], case.scale, workspace=workspace,
                                          **opts)
    torch.cuda.synchronize()
    return out.cpu(), ref.cpu(), (k1.cpu(), v1.cpu()), (k2.cpu(), v2.cpu())


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,G,S", [(128, 4, 16), (64, 1, 16), (128, 8, 32), (64, 2, 8), (128, 16, 16)])
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("split", [64, 128, None])
def test_fused_equals_write_then_decode(cuda_lib, dtype, D, G, S, kernel, split):
    pa = cuda_lib
    case = _case(dtype, 2 * G, 2, D, S, [0, 1, S - 1, S, 100, 777], seed=D + G + S)
    out, ref, pools_a, pools_b = _both(pa, case, workspace="auto" if split else None, decode_kernel=kernel,
                                       partition_tokens=split or 0)
    assert torch.equal(bits(out), bits(ref))
    assert torch.equal(bits(pools_a[0]), bits(pools_b[0])) and torch.equal(bits(pools_a[1]), bits(pools_b[1]))
    assert pa.device_error_flags() == 0


def test_fused_matches_oracle_on_the_serving_batch(cuda_lib):
    pa = cuda_lib
    case = W.llama_decode()
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    out = pa.paged_attention_decode_fused(case.q.cuda(), case.k_new.cuda(), case.v_new.cuda(),
                                          case.slot_mapping.cuda(), dk, dv, case.block_table.cuda(),
                                          case.context_lens.cuda(), case.scale).cpu()
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    rows = [(b, h) for b in range(0, 64, 3) for h in (0, 5)]
    ref = oracle.paged_decode_rows(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale, rows)
    for (b, h), r in ref.items():
        err = np.abs(out[b, 4 * h:4 * h + 4].double().numpy() - r).max()
        assert err <= 2e-2, (b, h, err)
    new_rows = dk.view(-1, 8, 128)[case.slot_mapping.cuda()].cpu()
    assert torch.equal(bits(new_rows), bits(case.k_new))


def test_negative_slot_writes_nothing_and_reads_the_pool(cuda_lib):
    pa = cuda_lib
    case = _case(torch.bfloat16, 8, 2, 128, 16, [40, 40], seed=3)
    slot = case.slot_mapping.clone()
    slot[0] = -1
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    kpool_before = dk.clone()
    lens = case.context_lens.clone()
    lens[0] -= 1  # sequence 0 attends over its history only
    out = pa.paged_attention_decode_fused(case.q.cuda(), case.k_new.cuda(), case.v_new.cuda(), slot.cuda(), dk, dv,
                                          case.block_table.cuda(), lens.cuda(), case.scale).cpu()
    assert pa.device_error_flags() == 0
    assert torch.equal(bits(dk.view(-1, 2, 128)[case.slot_mapping[0]].cpu()),
                       bits(kpool_before.view(-1, 2, 128)[case.slot_mapping[0]].cpu()))
    ref = oracle.paged_decode(case.q[:1], case.k_pool, case.v_pool, case.block_table[:1], lens[:1], case.scale)
    assert np.abs(out[:1].double().numpy() - ref).max() <= 2e-2


def test_slot_that_is_not_the_last_position_is_rejected(cuda_lib):
    pa = cuda_lib
    case = _case(torch.float16, 8, 2, 64, 16, [30, 30], seed=4)
    slot = case.slot_mapping.clone()
    slot[1] = slot[1] - 3  # a slot inside the history, not the last position
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    before = dk.clone()
    pa.paged_attention_decode_fused(case.q.cuda(), case.k_new.cuda(), case.v_new.cuda(), slot.cuda(), dk, dv,
                                    case.block_table.cuda(), case.context_lens.cuda(), case.scale)
    assert pa.device_error_flags() & pa.PA_DEVERR_SLOT
    assert torch.equal(bits(dk.view(-1, 2, 64)[slot[1]].cpu()), bits(before.view(-1, 2, 64)[slot[1]].cpu()))
    pa.set_checked_mode(True)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.paged_attention_decode_fused(case.q.cuda(), case.k_new.cuda(), case.v_new.cuda(), slot.cuda(), dk, dv,
                                        case.block_table.cuda(), case.context_lens.cuda(), case.scale)
    assert ei.value.status == pa.PA_ERANGE
