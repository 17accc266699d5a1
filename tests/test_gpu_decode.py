"""GPU parity: paged_kv_write, copy_blocks, paged_attention_decode (single pass and split-K) and
the log-sum-exp merge, each through the C ABI, against the fp64 CPU oracle on the same seeded
inputs.  Writes and copies must be bit-exact; attention within 2e-2 (bf16/fp16 I/O) or 1e-5
(fp32 I/O) max abs error."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.float16: 2e-2, torch.bfloat16: 2e-2}
DTYPES = [torch.bfloat16, torch.float16, torch.float32]


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, dtype, what=""):
    got = gpu.detach().double().cpu().numpy()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= TOL[dtype], f"{what}: max abs err {err} > {TOL[dtype]}"
    return err


@pytest.fixture(autouse=True)
def _reset_checked_mode(cuda_lib):
    pa = cuda_lib
    yield
    pa.set_checked_mode(False)
    pa.device_error_flags(clear=True)


def run_decode(pa, case, q=None, lens=None, kp=None, vp=None, workspace="auto", **opts):
    q = case.q if q is None else q
    lens = case.context_lens if lens is None else lens
    kp = case.k_pool.cuda() if kp is None else kp
    vp = case.v_pool.cuda() if vp is None else vp
    out = pa.paged_attention_decode(q.cuda(), kp, vp, case.block_table.cuda(), lens.cuda(), case.scale,
                                    workspace=workspace, **opts)
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------------------------------------
# bit-copy kernels
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("Hkv,D,S", [(2, 64, 16), (8, 128, 16), (8, 128, 32), (12, 64, 16), (1, 64, 1)])
def test_kv_write_bit_exact(cuda_lib, dtype, Hkv, D, S):
    pa = cuda_lib
    gen = torch.Generator().manual_seed(100 + Hkv + D + S)
    NB = 37
    kp = W.sentinel_pool(NB, S, Hkv, D, dtype)
    vp = W.sentinel_pool(NB, S, Hkv, D, dtype)
    T = min(NB * S, 300)
    slots = torch.randperm(NB * S, generator=gen)[:T].to(torch.int64)
    slots[::7] = -1
    kn = W.randn(gen, (T, Hkv, D), dtype)
    vn = W.randn(gen, (T, Hkv, D), dtype)
    ref_k, ref_v = oracle.paged_kv_write(kp, vp, kn, vn, slots)
    dk, dv = kp.cuda(), vp.cuda()
    pa.paged_kv_write(kn.cuda(), vn.cuda(), slots.cuda(), dk, dv)
    torch.cuda.synchronize()
    assert torch.equal(bits(dk.cpu()), bits(ref_k))
    assert torch.equal(bits(dv.cpu()), bits(ref_v))
    assert pa.device_error_flags() == 0


def test_kv_write_empty_and_out_of_range_slot(cuda_lib):
    pa = cuda_lib
    kp = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pa.paged_kv_write(torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                      torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda"),
                      torch.zeros(0, dtype=torch.int64, device="cuda"), kp, vp)
    kn = torch.ones((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([5, 4 * 16 + 3], dtype=torch.int64, device="cuda")  # second is past the pool
    pa.paged_kv_write(kn, kn, slots, kp, vp)
    assert pa.device_error_flags() & pa.PA_DEVERR_SLOT
    assert float(kp.view(-1, 2, 64)[5].float().min()) == 1.0
    assert float(kp.float().sum()) == 2 * 64  # nothing else written
    pa.set_checked_mode(True)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.paged_kv_write(kn, kn, slots, kp, vp)
    assert ei.value.status == pa.PA_ERANGE
    with pytest.raises(pa.PagedAttnError):
        pa.paged_kv_write(kn, kn, torch.tensor([3, 3], dtype=torch.int64, device="cuda"), kp, vp)


@pytest.mark.parametrize("dtype", DTYPES)
def test_copy_blocks_bit_exact(cuda_lib, dtype):
    pa = cuda_lib
    gen = torch.Generator().manual_seed(7)
    kp = W.randn(gen, (40, 32, 8, 128), dtype)
    vp = W.randn(gen, (40, 32, 8, 128), dtype)
    pairs = torch.tensor([[1, 30], [2, 31], [1, 33], [39, 0]], dtype=torch.int64)
    ref_k, ref_v = oracle.copy_blocks(kp, vp, pairs)
    dk, dv = kp.cuda(), vp.cuda()
    pa.copy_blocks(dk, dv, pairs.cuda())
    torch.cuda.synchronize()
    assert torch.equal(bits(dk.cpu()), bits(ref_k)) and torch.equal(bits(dv.cpu()), bits(ref_v))


def test_copy_blocks_bad_pair_is_flagged_not_faulted(cuda_lib):
    pa = cuda_lib
    kp = torch.zeros((4, 16, 2, 64), dtype=torch.float16, device="cuda")
    vp = torch.zeros_like(kp)
    kp[1] = 1
    pa.copy_blocks(kp, vp, torch.tensor([[1, 2], [1, 9]], dtype=torch.int64, device="cuda"))
    assert pa.device_error_flags() & pa.PA_DEVERR_COPY_PAIR
    assert float(kp[2].float().min()) == 1.0
    pa.set_checked_mode(True)
    with pytest.raises(pa.PagedAttnError):
        pa.copy_blocks(kp, vp, torch.tensor([[1, 2], [3, 2]], dtype=torch.int64, device="cuda"))


# ---------------------------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------------------------

def test_tiny_workload_both_steps(cuda_lib):
    pa = cuda_lib
    t = W.tiny_decode()
    dk, dv = t["k_pool"].cuda(), t["v_pool"].cuda()
    table, scale = t["block_table"].cuda(), t["scale"]
    out0 = pa.paged_attention_decode(t["q0"].cuda(), dk, dv, table, t["lens0"].cuda(), scale)
    ref0 = oracle.paged_decode(t["q0"], t["k_pool"], t["v_pool"], t["block_table"], t["lens0"], scale)
    assert_close(out0, ref0, torch.float32, "step 1")
    pa.paged_kv_write(t["k_new"].cuda(), t["v_new"].cuda(), t["slot_mapping"].cuda(), dk, dv)
    kp1, vp1 = oracle.paged_kv_write(t["k_pool"], t["v_pool"], t["k_new"], t["v_new"], t["slot_mapping"])
    torch.cuda.synchronize()
    assert torch.equal(bits(dk.cpu()), bits(kp1)) and torch.equal(bits(dv.cpu()), bits(vp1))
    out1 = pa.paged_attention_decode(t["q1"].cuda(), dk, dv, table, t["lens1"].cuda(), scale)
    ref1 = oracle.paged_decode(t["q1"], kp1, vp1, t["block_table"], t["lens1"], scale)
    assert_close(out1, ref1, torch.float32, "step 2")
    assert pa.device_error_flags() == 0


def _ragged_case(dtype, Hq, Hkv, D, S, lens, seed, NB=None):
    need = sum(W.ceil_div(n + 1, S) for n in lens)
    NB = NB or need + 7
    maxb = max(1, max(W.ceil_div(n + 1, S) for n in lens))
    return W.decode_case(f"ragged_{seed}", seed, lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, block_size=S,
                         dtype=dtype, num_blocks=NB, max_blocks_per_seq=maxb + 2)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("S", [8, 16, 32])
@pytest.mark.parametrize("part", [0, 64, 128, "none"])
@pytest.mark.parametrize("kernel", [0, 1])
def test_decode_shapes_and_partitions(cuda_lib, dtype, D, G, S, part, kernel):
    """kernel 0 = automatic choice (tensor-core path for bf16/fp16 with block_size % 16 == 0),
    1 = CUDA-core path forced.  part 64 gives 9-19 partitions per row, 128 gives 4-9 (workspace +
    merge kernel)."""
    pa = cuda_lib
    Hkv = 2
    lens = [0, 1, S - 1, S, S + 1, 3 * S + 5, 200, 517]  # history before the new token
    case = _ragged_case(dtype, Hkv * G, Hkv, D, S, lens, seed=D * 31 + G * 7 + S)
    ws = None if part == "none" else "auto"
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv, workspace=ws, decode_kernel=kernel,
                     partition_tokens=0 if part == "none" else part)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, dtype, f"{dtype} D{D} G{G} S{S} part{part} kernel{kernel}")
    assert pa.device_error_flags() == 0


# history lengths of a ragged batch: empty, single-token, block-aligned and long sequences next to
# each other, so that partitions end inside and at the end of blocks and long sequences split into
# many partitions
RAGGED_HIST = [0, 3000, 0, 15, 16, 1, 2047, 0, 5, 700, 4000, 31, 32, 33, 1500, 0, 2, 1023, 1024, 1025]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("part", [0, 16, 64, 512])
def test_decode_on_a_ragged_batch_with_empty_sequences(cuda_lib, dtype, part):
    """The split-K tensor-core decode against the oracle.  Sequences with history 0 are given
    context 0 (zeros out); part 16 gives 16-token partitions, so long sequences spread over hundreds
    of partitions (the one-CTA-per-row merge)."""
    pa = cuda_lib
    case = _ragged_case(dtype, 32, 8, 128, 16, RAGGED_HIST, seed=21 + part)
    lens = (case.context_lens - 1).clamp(min=0)  # history only: the new tokens are not written here
    out = run_decode(pa, case, lens=lens, partition_tokens=part)
    ref = oracle.paged_decode(case.q, case.k_pool, case.v_pool, case.block_table, lens, case.scale)
    assert_close(out, ref, dtype, f"part {part}")
    empty = (lens == 0).nonzero().flatten()
    assert torch.equal(out.cpu()[empty].float(), torch.zeros_like(out.cpu()[empty].float()))
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("G,D", [(1, 64), (2, 128), (4, 128), (8, 128), (8, 64), (16, 128), (16, 64)])
def test_ragged_batch_other_groups_and_head_dims(cuda_lib, G, D):
    """The ragged batch with 128-token partitions for every query-group size and head_dim."""
    pa = cuda_lib
    Hkv = 4
    case = _ragged_case(torch.bfloat16, Hkv * G, Hkv, D, 32, RAGGED_HIST, seed=40 + G * 3 + D)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv, partition_tokens=128)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, torch.bfloat16, f"G{G} D{D}")
    assert pa.device_error_flags() == 0


def test_split_decode_is_deterministic_and_stale_workspace_safe(cuda_lib):
    """Two calls on one workspace give the same bits, also after the workspace was filled with NaN
    and after a call on a different batch (no state is carried from call to call)."""
    pa = cuda_lib
    case = _ragged_case(torch.bfloat16, 32, 8, 128, 16, RAGGED_HIST, seed=23)
    other = _ragged_case(torch.bfloat16, 32, 8, 128, 16, list(reversed(RAGGED_HIST)), seed=24)
    nbytes = pa.decode_workspace_size(len(RAGGED_HIST), case.block_table.stride(0), 16, 32, 8, 128,
                                      partition_tokens=64)
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)
    lens = (case.context_lens - 1).clamp(min=0)  # history only: the new tokens are not written here
    out1 = run_decode(pa, case, lens=lens, workspace=ws, partition_tokens=64).cpu()
    run_decode(pa, other, lens=(other.context_lens - 1).clamp(min=0), workspace=ws, partition_tokens=64)
    out2 = run_decode(pa, case, lens=lens, workspace=ws, partition_tokens=64).cpu()
    assert torch.equal(bits(out1), bits(out2))
    assert torch.isfinite(out1.float()).all()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("part", [0, 64, "none"])
@pytest.mark.parametrize("kernel", [0, 1])
def test_decode_group_of_16_query_heads(cuda_lib, dtype, D, part, kernel):
    """16 query heads per KV head: both row halves of the tensor-core kernel's mma tile hold
    heads (and the CUDA-core path, kernel 1 or fp32, its largest query group)."""
    pa = cuda_lib
    ws = None if part == "none" else "auto"
    lens = [0, 1, 15, 16, 17, 200, 517, 1300]
    case = _ragged_case(dtype, 32, 2, D, 16, lens, seed=D + 16)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv, workspace=ws, decode_kernel=kernel,
                     partition_tokens=0 if part == "none" else part)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, dtype, f"G16 {dtype} D{D} part{part} kernel{kernel}")
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_token_context_returns_v_exactly(cuda_lib, dtype):
    pa = cuda_lib
    case = _ragged_case(dtype, 32, 8, 128, 16, [0, 0, 0], seed=5)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv).cpu()
    want = case.v_new.repeat_interleave(4, dim=1)
    assert torch.equal(bits(out.contiguous()), bits(want.contiguous()))


def test_empty_context_gives_zeros(cuda_lib):
    pa = cuda_lib
    case = _ragged_case(torch.bfloat16, 8, 2, 64, 16, [5, 9], seed=6)
    lens = torch.tensor([0, 9], dtype=torch.int32)  # history only: the new tokens are not written here
    out = run_decode(pa, case, lens=lens).cpu()
    assert torch.equal(out[0].float(), torch.zeros_like(out[0].float()))
    ref = oracle.paged_decode(case.q[1:], case.k_pool, case.v_pool, case.block_table[1:], lens[1:], case.scale)
    assert_close(out[1:], ref, torch.bfloat16)


def test_paged_read_is_bit_identical_under_block_relabelling(cuda_lib):
    """The reduction order depends only on logical positions, so relabelling physical blocks gives
    the same bits (nanoserve Day 19: the paged read equals the gather)."""
    pa = cuda_lib
    case = _ragged_case(torch.bfloat16, 32, 8, 128, 16, [700, 1500, 33], seed=8, NB=300)
    out_a = run_decode(pa, case).cpu()
    perm = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    kp2 = torch.empty_like(case.k_pool)
    vp2 = torch.empty_like(case.v_pool)
    kp2[inv] = case.k_pool
    vp2[inv] = case.v_pool
    table2 = torch.where(case.block_table >= 0, inv[case.block_table.clamp(min=0).long()].to(torch.int32),
                         case.block_table)
    out_b = pa.paged_attention_decode(case.q.cuda(), kp2.cuda(), vp2.cuda(), table2.cuda(),
                                      case.context_lens.cuda(), case.scale).cpu()
    assert torch.equal(bits(out_a), bits(out_b))


def test_bad_block_id_is_flagged_and_masked(cuda_lib):
    pa = cuda_lib
    case = _ragged_case(torch.float16, 8, 2, 64, 16, [40, 40], seed=9)
    lens = case.context_lens - 1  # history only: the new tokens are not written here
    table = case.block_table.clone()
    table[0, 1] = case.num_blocks + 1000  # out of range inside sequence 0's context
    out = pa.paged_attention_decode(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(), table.cuda(),
                                    lens.cuda(), case.scale).cpu()
    assert pa.device_error_flags() & pa.PA_DEVERR_BLOCK_ID
    # sequence 1 is unaffected; sequence 0 stays finite (its bad block is skipped)
    assert torch.isfinite(out.float()).all()
    ref = oracle.paged_decode(case.q[1:], case.k_pool, case.v_pool, case.block_table[1:], lens[1:], case.scale)
    assert_close(out[1:], ref, torch.float16)
    pa.set_checked_mode(True)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.paged_attention_decode(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(), table.cuda(),
                                  lens.cuda(), case.scale)
    assert ei.value.status == pa.PA_ERANGE


def test_nan_in_context_propagates_like_the_definition(cuda_lib):
    """A NaN key inside the context makes the two-pass softmax NaN; the kernel must not drop it."""
    pa = cuda_lib
    case = _ragged_case(torch.bfloat16, 8, 2, 64, 16, [100, 100], seed=12)
    lens = case.context_lens - 1
    out = run_decode(pa, case, lens=lens).cpu()  # position 100 (unwritten, NaN) is outside both contexts
    assert torch.isfinite(out.float()).all()
    out_nan = run_decode(pa, case, lens=lens + 1).cpu()  # now the NaN row is inside both contexts
    assert torch.isnan(out_nan.float()).all()


def test_tensor_core_path_refuses_unsupported_shapes(cuda_lib):
    pa = cuda_lib
    for dtype, S in ((torch.float32, 16), (torch.bfloat16, 8)):
        case = _ragged_case(dtype, 8, 2, 64, S, [20], seed=13)
        with pytest.raises(pa.PagedAttnError) as ei:
            run_decode(pa, case, decode_kernel=2)
        assert ei.value.status == pa.PA_EUNSUPPORTED


@pytest.mark.parametrize("kernel", [1, 2])
def test_both_kernels_agree_on_the_serving_shape(cuda_lib, kernel):
    """CUDA-core and tensor-core decode on a reduced serving batch (8 sequences, 512-4096 tokens)."""
    pa = cuda_lib
    lens = W.llama_context_lens()[:8]
    case = _ragged_case(torch.bfloat16, 32, 8, 128, 16, [n - 1 for n in lens], seed=14)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv, decode_kernel=kernel)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, torch.bfloat16, f"kernel {kernel}")


def test_workspace_too_small_is_rejected(cuda_lib):
    pa = cuda_lib
    case = _ragged_case(torch.bfloat16, 8, 2, 64, 16, [2000], seed=10)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.paged_attention_decode(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                                  case.block_table.cuda(), case.context_lens.cuda(), case.scale,
                                  workspace=torch.empty(64, dtype=torch.uint8, device="cuda"), partition_tokens=128)
    assert ei.value.status == pa.PA_EWORKSPACE


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,many", [(128, False), (128, True), (64, True)])
def test_lse_merge_matches_oracle_merge(cuda_lib, dtype, D, many):
    """The standalone merge against the oracle's; `many` gives 40 partitions (the one-CTA-per-row
    merge for rows of 16 or more partitions), some of them empty."""
    pa = cuda_lib
    rng = np.random.default_rng(11 + D + many)
    H, n = 6, 300
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((n, H, D))
    k[rng.choice(n, 4, replace=False)] *= 8
    v = rng.standard_normal((n, H, D))
    if many:
        cuts = [0, 0] + sorted(int(c) for c in rng.choice(np.arange(1, n), 37, replace=False)) + [n, n]
    else:
        cuts = [0, 0, 50, 51, 51, 200, 300]  # includes empty partitions
    parts = oracle.partition_partials(q, k, v, 0.3, list(zip(cuts[:-1], cuts[1:])))
    P = len(parts)
    log2e = 1.0 / math.log(2.0)
    pm = np.stack([p[0] for p in parts], axis=1) * log2e           # [H, P] in the log2 domain
    pl = np.stack([p[1] for p in parts], axis=1)
    pacc = np.stack([p[2] for p in parts], axis=1)                 # [H, P, D]
    out = pa.paged_attention_lse_merge(torch.tensor(pm, dtype=torch.float32).cuda(),
                                       torch.tensor(pl, dtype=torch.float32).cuda(),
                                       torch.tensor(pacc, dtype=torch.float32).cuda(), out_dtype=dtype)
    torch.cuda.synchronize()
    assert P == (40 if many else 6)
    assert_close(out, oracle.lse_merge(parts), dtype, "merge")


# ---------------------------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("batch", W.GPT2_BATCHES)
@pytest.mark.parametrize("context", W.GPT2_CONTEXTS)
def test_gpt2_sweep_cell(cuda_lib, batch, context):
    pa = cuda_lib
    case = W.gpt2_decode(batch, context, layer=batch % 12)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv)
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, torch.float16, case.name)


@pytest.mark.slow
def test_llama_serving_decode_full(cuda_lib):
    """Llama-3-8B-shaped serving step at full size, in the launch configuration bench.py times."""
    pa = cuda_lib
    case = W.llama_decode()
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv).cpu()
    # the write: every new row landed, bit-exact
    flat_k = dk.view(-1, 8, 128)[case.slot_mapping.cuda()].cpu()
    assert torch.equal(bits(flat_k), bits(case.k_new))
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    ref = oracle.paged_decode(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale)
    assert_close(out, ref, torch.bfloat16, "llama")
    assert pa.device_error_flags() == 0


@pytest.mark.slow
def test_long_context_split_k_full(cuda_lib):
    """Long-context decode (32K-128K tokens, peaked rows) against the oracle on sampled KV heads,
    and split-K against the unsplit kernel on the same inputs."""
    pa = cuda_lib
    case = W.long_context_decode()
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = run_decode(pa, case, kp=dk, vp=dv).cpu()
    kp1, vp1 = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    rows = [(b, h) for b in range(4) for h in (b % 8, 7 - b % 8)]
    ref = oracle.paged_decode_rows(case.q, kp1, vp1, case.block_table, case.context_lens, case.scale, rows)
    for (b, h), r in ref.items():
        assert_close(out[b, 4 * h:4 * h + 4], r, torch.bfloat16, f"long b{b} h{h}")
    out_nosplit = run_decode(pa, case, kp=dk, vp=dv, workspace=None).cpu()
    err = (out.double() - out_nosplit.double()).abs().max().item()
    assert err <= 2e-2
