"""GPU parity for causal chunked prefill over a paged history, and for the copy-on-write arm
(copy_blocks fork, then the write, then the prefill) against the unshared-copy oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.float16: 2e-2, torch.bfloat16: 2e-2}
DTYPES = [torch.bfloat16, torch.float16, torch.float32]


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype, what=""):
    g = got.detach().double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref).max() if ref.size else 0.0
    assert err <= TOL[dtype], f"{what}: max abs err {err} > {TOL[dtype]}"


@pytest.fixture(autouse=True)
def _reset_checked_mode(cuda_lib):
    yield
    cuda_lib.set_checked_mode(False)
    cuda_lib.device_error_flags(clear=True)


def run_case(pa, case, kernel=0):
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    if case.copy_pairs.numel():
        pa.copy_blocks(dk, dv, case.copy_pairs.cuda())
    if case.slot_mapping.numel():
        pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = pa.paged_attention_prefill(case.q.cuda(), case.query_start_loc.cuda(), dk, dv,
                                     case.block_table.cuda(), case.context_lens.cuda(), case.scale,
                                     prefill_kernel=kernel)
    torch.cuda.synchronize()
    return out.cpu(), dk, dv


def oracle_pools(case):
    kp, vp = case.k_pool, case.v_pool
    if case.copy_pairs.numel():
        kp, vp = oracle.copy_blocks(kp, vp, case.copy_pairs)
    return oracle.paged_kv_write(kp, vp, case.k_new, case.v_new, case.slot_mapping)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("S", [16, 32])
@pytest.mark.parametrize("kernel", [0, 1])
def test_prefill_ragged_chunks(cuda_lib, dtype, D, G, S, kernel):
    """kernel 0 = automatic (tcgen05 path for bf16/fp16, CUDA cores for fp32), 1 = CUDA cores."""
    pa = cuda_lib
    case = W.varlen_prefill(D + G + S, hist_lens=[0, 5, 40, 17, 130, 0, 300], chunk_lens=[9, 0, 23, 1, 70, 64, 200],
                            block_size=S, n_q_heads=2 * G, n_kv_heads=2, head_dim=D, dtype=dtype,
                            num_blocks=96)
    out, _, _ = run_case(pa, case, kernel=kernel)
    kp, vp = oracle_pools(case)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens,
                               case.scale)
    idx = sorted(res)
    assert len(idx) == case.q.shape[0]
    assert_close(out[idx], np.stack([res[i] for i in idx]), dtype, f"prefill {dtype} D{D} G{G} S{S} k{kernel}")
    assert pa.device_error_flags() == 0


def _peak_keys(case, offsets, factor):
    """Scale the keys of context positions p with p % 128 in ``offsets`` (history keys in the pool,
    chunk keys in k_new) by ``factor``, in place."""
    S = case.block_size
    qsl = case.query_start_loc.tolist()
    lens = case.context_lens.tolist()
    for b, n in enumerate(lens):
        m = qsl[b + 1] - qsl[b]
        for p in range(n):
            if p % 128 not in offsets:
                continue
            if p < n - m:
                blk = int(case.block_table[b, p // S])
                case.k_pool[blk, p % S] = (case.k_pool[blk, p % S].float() * factor).to(case.dtype)
            else:
                r = qsl[b] + p - (n - m)
                case.k_new[r] = (case.k_new[r].float() * factor).to(case.dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("G,D", [(4, 128), (2, 64)])
def test_prefill_peaked_keys_in_second_half_of_tiles(cuda_lib, dtype, G, D):
    """Keys in the second 64 keys of 128-key tiles scaled x16: within a tile the scores of keys
    64..127 exceed those of keys 0..63 by far more than 2^8 in the exponent's base-2 units, so the
    softmax moves its stabilising maximum after the first half's probabilities are already stored
    (and, at other rows and tiles, before); every output against the oracle."""
    pa = cuda_lib
    case = W.varlen_prefill(77 + G + D, hist_lens=[300, 0, 190, 520], chunk_lens=[96, 200, 33, 128],
                            block_size=16, n_q_heads=2 * G, n_kv_heads=2, head_dim=D, dtype=dtype,
                            num_blocks=160)
    _peak_keys(case, {71, 100, 127}, 16.0)
    out, _, _ = run_case(pa, case, kernel=0)
    kp, vp = oracle_pools(case)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens,
                               case.scale)
    idx = sorted(res)
    assert len(idx) == case.q.shape[0]
    assert_close(out[idx], np.stack([res[i] for i in idx]), dtype, f"peaked {dtype} G{G} D{D}")
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("G,D", [(4, 128), (8, 64)])
def test_prefill_many_items_per_cta(cuda_lib, G, D):
    """More (64-token query block, KV head) items than SMs, so every CTA of the tcgen05 kernel
    walks several items in turn (Q reloaded, O handed over between items) across ragged chunks,
    empty chunks and chunk boundaries inside an item; all outputs against the oracle."""
    pa = cuda_lib
    rng = np.random.default_rng(31 + G + D)
    B = 48
    hist = [int(x) for x in rng.integers(0, 400, B)]
    chunks = [int(x) for x in rng.integers(0, 180, B)]
    chunks[3] = 0
    chunks[7] = 1
    Hkv = 8
    need = sum(W.ceil_div(h + c, 16) for h, c in zip(hist, chunks))
    case = W.varlen_prefill(4242 + G, hist_lens=hist, chunk_lens=chunks, block_size=16, n_q_heads=Hkv * G,
                            n_kv_heads=Hkv, head_dim=D, dtype=torch.bfloat16, num_blocks=need + 9)
    assert sum(chunks) // (256 // G) * Hkv > 2 * 152  # several items per CTA
    out, _, _ = run_case(pa, case, kernel=0)
    kp, vp = oracle_pools(case)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens, case.scale)
    idx = sorted(res)
    assert len(idx) == case.q.shape[0]
    assert_close(out[idx], np.stack([res[i] for i in idx]), torch.bfloat16, f"G{G} D{D}")
    assert pa.device_error_flags() == 0


@pytest.mark.parametrize("kernel", [0, 1])
def test_prefill_cow_arm_small_equals_unshared_copy(cuda_lib, kernel):
    """Copy-on-write fork of a shared partial block: the forked sequences attend exactly like
    sequences that never shared (JuliaPagedAttn README, "Copy-on-Write")."""
    pa = cuda_lib
    case = W.small_prefill(21, batch=6, prefix=100, suffix_max=40, chunk=24, block_size=32, n_q_heads=32,
                           n_kv_heads=8, head_dim=128, dtype=torch.bfloat16, num_blocks=80,
                           suffix_in_cache=False)
    assert case.copy_pairs.shape[0] == 5
    out, _, _ = run_case(pa, case, kernel=kernel)
    qsl = case.query_start_loc.tolist()
    for b in range(6):
        k_l, v_l = case.extra["logical"][b]
        ref = oracle.causal_attention_contiguous(oracle.to_f64(case.q[qsl[b]:qsl[b + 1]]), oracle.to_f64(k_l),
                                                 oracle.to_f64(v_l), case.scale)
        assert_close(out[qsl[b]:qsl[b + 1]], ref, torch.bfloat16, f"cow seq {b}")
    # GPU against GPU: the same sequences laid out with private prefix copies give the same bits
    S = 32
    lens = case.context_lens.tolist()
    table = torch.full_like(case.block_table, -1)
    kp = W.sentinel_pool(80, S, 8, 128, torch.bfloat16)
    vp = W.sentinel_pool(80, S, 8, 128, torch.bfloat16)
    nxt = 0
    for b in range(6):
        nb = W.ceil_div(lens[b], S)
        table[b, :nb] = torch.arange(nxt, nxt + nb, dtype=torch.int32)
        nxt += nb
        k_l, v_l = case.extra["logical"][b]
        sl = W.slots_for(table[b], range(lens[b]), S)
        kp.view(-1, 8, 128)[sl] = k_l
        vp.view(-1, 8, 128)[sl] = v_l
    out2 = pa.paged_attention_prefill(case.q.cuda(), case.query_start_loc.cuda(), kp.cuda(), vp.cuda(),
                                      table.cuda(), case.context_lens.cuda(), case.scale, prefill_kernel=kernel).cpu()
    assert torch.equal(bits(out), bits(out2))


@pytest.mark.parametrize("kernel", [1, 2])
def test_prefill_bad_block_id_is_flagged(cuda_lib, kernel):
    pa = cuda_lib
    case = W.varlen_prefill(4, hist_lens=[40, 40], chunk_lens=[24, 24], block_size=16, n_q_heads=8, n_kv_heads=2,
                            head_dim=128, dtype=torch.bfloat16, num_blocks=16)
    table = case.block_table.clone()
    table[0, 1] = 999
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = pa.paged_attention_prefill(case.q.cuda(), case.query_start_loc.cuda(), dk, dv, table.cuda(),
                                     case.context_lens.cuda(), case.scale, prefill_kernel=kernel).cpu()
    assert pa.device_error_flags() & pa.PA_DEVERR_BLOCK_ID
    kp, vp = oracle_pools(case)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens,
                               case.scale, seqs=[1])
    idx = sorted(res)
    assert_close(out[idx], np.stack([res[i] for i in idx]), torch.bfloat16, "unaffected sequence")


def test_prefill_tensor_core_refuses_unsupported(cuda_lib):
    pa = cuda_lib
    case = W.varlen_prefill(5, hist_lens=[3], chunk_lens=[5], block_size=8, n_q_heads=4, n_kv_heads=2,
                            head_dim=64, dtype=torch.bfloat16, num_blocks=4)
    with pytest.raises(pa.PagedAttnError) as ei:
        run_case(pa, case, kernel=2)
    assert ei.value.status == pa.PA_EUNSUPPORTED


def test_prefill_bad_query_start_loc_is_flagged(cuda_lib):
    pa = cuda_lib
    case = W.varlen_prefill(3, hist_lens=[4, 4], chunk_lens=[8, 8], block_size=16, n_q_heads=8, n_kv_heads=2,
                            head_dim=64, dtype=torch.float16, num_blocks=8)
    lens = torch.tensor([6, 12], dtype=torch.int32)  # chunk of sequence 0 longer than its context
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pa.paged_kv_write(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), dk, dv)
    out = pa.paged_attention_prefill(case.q.cuda(), case.query_start_loc.cuda(), dk, dv,
                                     case.block_table.cuda(), lens.cuda(), case.scale)
    torch.cuda.synchronize()
    assert pa.device_error_flags() & pa.PA_DEVERR_QUERY_LOC
    assert torch.isfinite(out.float()).all()
    pa.set_checked_mode(True)
    with pytest.raises(pa.PagedAttnError):
        pa.paged_attention_prefill(case.q.cuda(), case.query_start_loc.cuda(), dk, dv, case.block_table.cuda(),
                                   lens.cuda(), case.scale)


def _sampled_check(case, out, seqs, rows_per_seq):
    kp, vp = oracle_pools(case)
    m = W.PREFILL_CHUNK
    queries = sorted(set([0, 1, m // 2, m - 2, m - 1] + list(range(0, m, max(1, m // rows_per_seq)))))
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens,
                               case.scale, seqs=seqs, queries=queries)
    idx = sorted(res)
    assert_close(out[idx], np.stack([res[i] for i in idx]), torch.bfloat16, case.name)


@pytest.mark.slow
@pytest.mark.parametrize("kernel", [1, 2])
def test_prefill_shared_prefix_full(cuda_lib, kernel):
    """Chunked prefill, 128 sequences over a 1024-token shared prefix: sampled rows vs the oracle
    (kernel 1 = CUDA cores, 2 = tcgen05, the launch configuration bench.py times)."""
    pa = cuda_lib
    case = W.prefill_cow()
    out, _, _ = run_case(pa, case, kernel=kernel)
    assert torch.isfinite(out.float()).all()
    _sampled_check(case, out, seqs=[0, 1, 37, 64, 100, 127], rows_per_seq=16)


@pytest.mark.slow
def test_prefill_cow_fork_full(cuda_lib):
    """The copy-on-write arm at full size: a 1000-token shared prefix ends inside block 31; every
    sequence's first write forks it (127 copies, one in-place write)."""
    pa = cuda_lib
    case = W.prefill_cow(cow_arm=True)
    assert case.copy_pairs.shape[0] == W.PREFILL_BATCH - 1
    out, dk, _ = run_case(pa, case)
    kp, _ = oracle_pools(case)
    # forked and written blocks are bit-exact
    touched = torch.unique(torch.cat([case.copy_pairs[:, 1], case.slot_mapping // 32]))
    assert torch.equal(bits(dk.cpu()[touched]), bits(kp[touched]))
    qsl = case.query_start_loc.tolist()
    for b in (0, 5, 77, 127):
        k_l, v_l = case.extra["logical"][b]
        rows = list(range(0, W.PREFILL_CHUNK, 17)) + [W.PREFILL_CHUNK - 1]
        q = oracle.to_f64(case.q[qsl[b]:qsl[b + 1]])
        ref = oracle.causal_attention_contiguous(q, oracle.to_f64(k_l), oracle.to_f64(v_l), case.scale)
        assert_close(out[qsl[b]:qsl[b + 1]][rows], ref[rows], torch.bfloat16, f"cow full seq {b}")


@pytest.mark.parametrize("kernel", [0, 1])
def test_mixed_decode_and_prefill_batch(cuda_lib, kernel):
    """The continuous-batching step: decode rows (1-query chunks at the last position) and prefill
    chunks of any length in one paged_attention_prefill launch; the decode rows also agree with
    paged_attention_decode on the same sequences."""
    pa = cuda_lib
    hist = [700, 0, 95, 1500, 33, 260, 1023]
    chunk = [1, 128, 1, 1, 64, 1, 200]
    case = W.varlen_prefill(99, hist_lens=hist, chunk_lens=chunk, block_size=16, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, dtype=torch.bfloat16, num_blocks=400)
    out, dk, dv = run_case(pa, case, kernel=kernel)
    kp, vp = oracle_pools(case)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table, case.context_lens, case.scale)
    idx = sorted(res)
    assert_close(out[idx], np.stack([res[i] for i in idx]), torch.bfloat16, f"mixed k{kernel}")
    # decode rows through the decode kernel
    qsl = case.query_start_loc.tolist()
    dec = [b for b, m in enumerate(chunk) if m == 1]
    qd = torch.stack([case.q[qsl[b]] for b in dec])
    od = pa.paged_attention_decode(qd.cuda(), dk, dv, case.block_table[dec].contiguous().cuda(),
                                   case.context_lens[dec].cuda(), case.scale).cpu()
    for i, b in enumerate(dec):
        assert (od[i].double() - out[qsl[b]].double()).abs().max().item() <= 2e-2
