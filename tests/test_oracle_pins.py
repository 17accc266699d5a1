"""Pins for the CPU oracle: it is checked here against facts fixed by the pages and by mathematics,
never against itself or the GPU path.

* single-token context returns V exactly; identical keys or scale 0 give the mean of V (closed
  forms of the softmax-weighted sum, JuliaPagedAttn README "Online Softmax");
* the single-pass online softmax equals the two-pass softmax (JuliaPagedAttn "Online Softmax");
* the paged read equals the contiguous-gather read and is invariant under relabelling physical
  blocks (nanoserve Day 19 "Why it matters": the fused read is identical to the gather);
* a copy-on-write fork gives the same attention as an unshared copy (JuliaPagedAttn
  "Copy-on-Write");
* GQA with the read-time repeat equals torch's fp64 scaled_dot_product_attention on explicitly
  repeated heads (nanoserve Day 19 "What I learned" item 4), for decode and causal prefill;
* pure-Python brute force (blocks walked one by one, math.exp) on the tiny workload;
* the log-sum-exp merge of any partition equals the unpartitioned result;
* the hand-worked example in tests/golden/hand_worked_decode.txt;
* planted mistakes (wrong GQA map, dropped scale, off-by-one causal bound, swapped slot
  arithmetic) each fail at least one of the pins above.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import paged_oracle as PO

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pool_from_logical(k_logical, table, S, NB, fill=float("nan")):
    """Place a contiguous [n, Hkv, D] history into a pool through a table (test-side placement)."""
    n, Hkv, D = k_logical.shape
    pool = torch.full((NB, S, Hkv, D), fill, dtype=k_logical.dtype)
    for j in range(n):
        pool[int(table[j // S]), j % S] = k_logical[j]
    return pool


def _sdpa(q, k, v, scale, mask=None):
    """torch fp64 SDPA. q [Hq, m, D], k/v [Hq, n, D]."""
    return torch.nn.functional.scaled_dot_product_attention(
        q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), attn_mask=mask, scale=scale).squeeze(0)


# ---------------------------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------------------------

def test_single_token_context_returns_v_exactly():
    gen = torch.Generator().manual_seed(1)
    S, Hq, Hkv, D, NB = 16, 8, 2, 64, 4
    k = torch.randn((1, Hkv, D), generator=gen, dtype=torch.float64)
    v = torch.randn((1, Hkv, D), generator=gen, dtype=torch.float64)
    table = torch.tensor([[3]], dtype=torch.int32)
    kp, vp = _pool_from_logical(k, table[0], S, NB), _pool_from_logical(v, table[0], S, NB)
    q = torch.randn((1, Hq, D), generator=gen, dtype=torch.float64) * 10
    out = oracle.paged_decode(q, kp, vp, table, torch.tensor([1]), 0.125)
    g = Hq // Hkv
    for h in range(Hq):
        assert np.array_equal(out[0, h], v[0, h // g].numpy())


@pytest.mark.parametrize("scale_zero", [False, True])
def test_identical_keys_or_zero_scale_give_mean_of_v(scale_zero):
    gen = torch.Generator().manual_seed(2)
    S, Hq, Hkv, D, NB, n = 16, 4, 2, 32, 8, 37
    if scale_zero:
        k = torch.randn((n, Hkv, D), generator=gen, dtype=torch.float64)
        scale = 0.0
    else:
        k = torch.randn((1, Hkv, D), generator=gen, dtype=torch.float64).repeat(n, 1, 1)
        scale = 0.3
    v = torch.randn((n, Hkv, D), generator=gen, dtype=torch.float64)
    table = torch.tensor([5, 1, 7], dtype=torch.int32)
    kp, vp = _pool_from_logical(k, table, S, NB), _pool_from_logical(v, table, S, NB)
    q = torch.randn((1, Hq, D), generator=gen, dtype=torch.float64)
    out = oracle.paged_decode(q, kp, vp, table[None], torch.tensor([n]), scale)
    mean = v.mean(dim=0).numpy()
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], mean[h // (Hq // Hkv)], rtol=0, atol=1e-13)


def test_empty_context_gives_zeros():
    kp = torch.full((2, 4, 1, 8), float("nan"), dtype=torch.float64)
    out = oracle.paged_decode(torch.ones((1, 2, 8)), kp, kp, torch.tensor([[-1]], dtype=torch.int32),
                              torch.tensor([0]), 1.0)
    assert np.array_equal(out, np.zeros((1, 2, 8)))


def test_hand_worked_example():
    fields = {}
    pools = {"pool_k": {}, "pool_v": {}}
    with open(os.path.join(GOLDEN, "hand_worked_decode.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(" ", 1)
            if key in pools:
                a, b, x, y = rest.split()
                pools[key][(int(a), int(b))] = [float(x), float(y)]
            else:
                fields[key] = rest
    S, D = int(fields["block_size"]), int(fields["head_dim"])
    kp = torch.zeros((3, S, 1, D), dtype=torch.float64)
    vp = torch.zeros((3, S, 1, D), dtype=torch.float64)
    for (blk, row), val in pools["pool_k"].items():
        kp[blk, row, 0] = torch.tensor(val)
    for (blk, row), val in pools["pool_v"].items():
        vp[blk, row, 0] = torch.tensor(val)
    table = torch.tensor([[int(x) for x in fields["table"].split()]], dtype=torch.int32)
    q = torch.tensor([[[float(x) for x in fields["query"].split()]]], dtype=torch.float64)
    out = oracle.paged_decode(q, kp, vp, table, torch.tensor([int(fields["context_len"])]),
                              float(fields["scale"]))
    e = math.e
    expect = [eval(fields["expect_0"], {"e": e}), eval(fields["expect_1"], {"e": e})]
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-15)
    # the same numbers through the single-pass form
    kc = oracle.gather_history(kp, table[0], 3, S)
    vc = oracle.gather_history(vp, table[0], 3, S)
    np.testing.assert_allclose(oracle.online_softmax_attention(q[0].numpy(), kc, vc, 1.0)[0], expect,
                               rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# algorithm identities
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("peaked", [False, True])
def test_online_softmax_equals_two_pass(peaked):
    rng = np.random.default_rng(3)
    H, D, n = 4, 16, 150
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((n, H, D))
    if peaked:
        k[rng.choice(n, 3, replace=False)] *= 8.0
    v = rng.standard_normal((n, H, D))
    a = oracle.online_softmax_attention(q, k, v, 0.25)
    b = oracle.softmax_attention(q, k, v, 0.25)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("cuts", [[0, 150], [0, 1, 150], [0, 16, 32, 33, 150], [0, 0, 70, 70, 150],
                                  list(range(0, 151, 10))])
def test_lse_merge_of_any_partition_equals_whole(cuts):
    rng = np.random.default_rng(4)
    H, D, n = 4, 16, 150
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((n, H, D))
    k[rng.choice(n, 2, replace=False)] *= 8.0
    v = rng.standard_normal((n, H, D))
    parts = oracle.partition_partials(q, k, v, 0.5, list(zip(cuts[:-1], cuts[1:])))
    np.testing.assert_allclose(oracle.lse_merge(parts), oracle.softmax_attention(q, k, v, 0.5),
                               rtol=0, atol=1e-12)


def test_paged_read_equals_contiguous_gather_and_is_permutation_invariant():
    gen = torch.Generator().manual_seed(5)
    S, Hq, Hkv, D, NB = 16, 8, 2, 32, 20
    lens = [1, 16, 17, 45]
    ks = [torch.randn((n, Hkv, D), generator=gen, dtype=torch.float64) for n in lens]
    vs = [torch.randn((n, Hkv, D), generator=gen, dtype=torch.float64) for n in lens]
    q = torch.randn((len(lens), Hq, D), generator=gen, dtype=torch.float64)
    maxb = 3

    def run(perm):
        table = torch.full((len(lens), maxb), -1, dtype=torch.int32)
        kp = torch.full((NB, S, Hkv, D), float("nan"), dtype=torch.float64)
        vp = kp.clone()
        pos = 0
        for b, n in enumerate(lens):
            nb = W.ceil_div(n, S)
            table[b, :nb] = torch.tensor(perm[pos:pos + nb], dtype=torch.int32)
            pos += nb
            for j in range(n):
                kp[int(table[b, j // S]), j % S] = ks[b][j]
                vp[int(table[b, j // S]), j % S] = vs[b][j]
        return oracle.paged_decode(q, kp, vp, table, torch.tensor(lens), 0.2)

    contiguous = run(list(range(NB)))
    shuffled = run([int(x) for x in torch.randperm(NB, generator=gen)])
    relabelled = run(list(reversed(range(NB))))
    assert np.array_equal(contiguous, shuffled)
    assert np.array_equal(contiguous, relabelled)
    # the gather path (contiguous history, then ordinary attention)
    for b, n in enumerate(lens):
        kr = np.repeat(ks[b].numpy(), Hq // Hkv, axis=1)
        vr = np.repeat(vs[b].numpy(), Hq // Hkv, axis=1)
        assert np.array_equal(contiguous[b], oracle.softmax_attention(q[b].numpy(), kr, vr, 0.2))


# ---------------------------------------------------------------------------------------------
# library special cases (torch SDPA, fp64, CPU)
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("Hq,Hkv", [(6, 6), (8, 2), (32, 8)])
def test_decode_matches_torch_sdpa(Hq, Hkv):
    gen = torch.Generator().manual_seed(6)
    S, D, NB = 16, 32, 40
    lens = [1, 33, 100]
    table = W.shuffled_block_tables(gen, NB, lens, S, 8)
    ks = [torch.randn((n, Hkv, D), generator=gen, dtype=torch.float64) for n in lens]
    vs = [torch.randn((n, Hkv, D), generator=gen, dtype=torch.float64) for n in lens]
    kp = torch.full((NB, S, Hkv, D), float("nan"), dtype=torch.float64)
    vp = kp.clone()
    for b, n in enumerate(lens):
        sl = W.slots_for(table[b], range(n), S)
        kp.view(-1, Hkv, D)[sl] = ks[b]
        vp.view(-1, Hkv, D)[sl] = vs[b]
    q = torch.randn((len(lens), Hq, D), generator=gen, dtype=torch.float64)
    out = oracle.paged_decode(q, kp, vp, table, torch.tensor(lens), 0.17)
    for b, n in enumerate(lens):
        kr = ks[b].repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)  # [Hq, n, D]
        vr = vs[b].repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)
        ref = _sdpa(q[b][:, None, :], kr, vr, 0.17)[:, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)


def test_prefill_matches_torch_sdpa_with_offset_causal_mask():
    case = W.varlen_prefill(7, hist_lens=[0, 5, 40, 17], chunk_lens=[9, 0, 23, 16], block_size=8,
                            n_q_heads=8, n_kv_heads=2, head_dim=16, dtype=torch.float64, num_blocks=40)
    kp, vp = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table,
                               case.context_lens, case.scale)
    g = case.n_q_heads // case.n_kv_heads
    qsl = case.query_start_loc.tolist()
    for b in range(4):
        m = qsl[b + 1] - qsl[b]
        if m == 0:
            continue
        n = int(case.context_lens[b])
        sl = W.slots_for(case.block_table[b], range(n), case.block_size)
        kc = kp.view(-1, 2, 16)[sl].repeat_interleave(g, dim=1).transpose(0, 1)
        vc = vp.view(-1, 2, 16)[sl].repeat_interleave(g, dim=1).transpose(0, 1)
        qb = case.q[qsl[b]:qsl[b + 1]].transpose(0, 1)  # [Hq, m, D]
        rows = torch.arange(m)[:, None] + (n - m)
        cols = torch.arange(n)[None, :]
        mask = cols <= rows  # boolean: True = attend
        ref = _sdpa(qb, kc, vc, case.scale, mask=mask).transpose(0, 1)
        for r in range(m):
            np.testing.assert_allclose(res[qsl[b] + r], ref[r].numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# brute force on the tiny workload
# ---------------------------------------------------------------------------------------------

def _brute_force_decode(q, k_pool, v_pool, table, lens, scale, Hq, Hkv):
    """Pure-Python loops: walk each sequence's blocks in order, token by token."""
    out = []
    g = Hq // Hkv
    S = len(k_pool[0])
    D = len(k_pool[0][0][0])
    for b, n in enumerate(lens):
        rows_k, rows_v = [], []
        lb = 0
        while len(rows_k) < n:
            phys = int(table[b][lb])
            for off in range(S):
                if len(rows_k) == n:
                    break
                rows_k.append(k_pool[phys][off])
                rows_v.append(v_pool[phys][off])
            lb += 1
        heads = []
        for h in range(Hq):
            kvh = h // g
            scores = [scale * sum(float(q[b][h][d]) * float(rows_k[j][kvh][d]) for d in range(D))
                      for j in range(n)]
            mx = max(scores)
            w = [math.exp(s - mx) for s in scores]
            tot = sum(w)
            heads.append([sum(w[j] * float(rows_v[j][kvh][d]) for j in range(n)) / tot for d in range(D)])
        out.append(heads)
    return np.array(out)


def test_brute_force_tiny_workload_both_steps():
    t = W.tiny_decode()
    out0 = oracle.paged_decode(t["q0"], t["k_pool"], t["v_pool"], t["block_table"], t["lens0"], t["scale"])
    bf0 = _brute_force_decode(t["q0"].tolist(), t["k_pool"].tolist(), t["v_pool"].tolist(),
                              t["block_table"].tolist(), t["lens0"].tolist(), t["scale"], 8, 2)
    np.testing.assert_allclose(out0, bf0, rtol=0, atol=1e-12)
    kp, vp = oracle.paged_kv_write(t["k_pool"], t["v_pool"], t["k_new"], t["v_new"], t["slot_mapping"])
    out1 = oracle.paged_decode(t["q1"], kp, vp, t["block_table"], t["lens1"], t["scale"])
    bf1 = _brute_force_decode(t["q1"].tolist(), kp.tolist(), vp.tolist(), t["block_table"].tolist(),
                              t["lens1"].tolist(), t["scale"], 8, 2)
    np.testing.assert_allclose(out1, bf1, rtol=0, atol=1e-12)
    assert np.isfinite(out0).all() and np.isfinite(out1).all()


# ---------------------------------------------------------------------------------------------
# bit-copy operations
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_write_round_trip_and_sentinels(dtype):
    gen = torch.Generator().manual_seed(8)
    NB, S, Hkv, D = 6, 4, 2, 8
    kp = torch.full((NB, S, Hkv, D), float("nan"), dtype=dtype)
    vp = kp.clone()
    T = 9
    slots = torch.randperm(NB * S, generator=gen)[:T].to(torch.int64)
    slots[3] = -1  # a token with no slot
    kn = torch.randn((T, Hkv, D), generator=gen).to(dtype)
    vn = torch.randn((T, Hkv, D), generator=gen).to(dtype)
    k2, v2 = oracle.paged_kv_write(kp, vp, kn, vn, slots)
    kf, vf = k2.view(-1, Hkv, D), v2.view(-1, Hkv, D)
    for t in range(T):
        if slots[t] >= 0:
            assert torch.equal(kf[slots[t]], kn[t]) and torch.equal(vf[slots[t]], vn[t])
    written = set(int(s) for s in slots if s >= 0)
    for s in range(NB * S):
        if s not in written:
            assert torch.isnan(kf[s].float()).all() and torch.isnan(vf[s].float()).all()
    assert torch.isnan(kp.float()).all()  # input untouched


def test_write_is_sequential_for_repeated_slots():
    kp = torch.zeros((2, 2, 1, 2))
    kn = torch.tensor([[[1.0, 1.0]], [[2.0, 2.0]]])
    k2, _ = oracle.paged_kv_write(kp, kp.clone(), kn, kn, torch.tensor([3, 3]))
    assert torch.equal(k2.view(-1, 1, 2)[3], kn[1])


def test_copy_blocks_bit_exact():
    gen = torch.Generator().manual_seed(9)
    kp = torch.randn((6, 4, 2, 8), generator=gen).to(torch.bfloat16)
    vp = torch.randn((6, 4, 2, 8), generator=gen).to(torch.bfloat16)
    k2, v2 = oracle.copy_blocks(kp, vp, torch.tensor([[1, 4], [2, 5]]))
    assert torch.equal(k2[4], kp[1]) and torch.equal(v2[5], vp[2])
    for blk in (0, 1, 2, 3):
        assert torch.equal(k2[blk], kp[blk]) and torch.equal(v2[blk], vp[blk])


def test_cow_fork_equals_unshared_copy():
    case = W.small_prefill(11, batch=5, prefix=44, suffix_max=20, chunk=12, block_size=16,
                           n_q_heads=4, n_kv_heads=2, head_dim=16, dtype=torch.float32,
                           num_blocks=64, suffix_in_cache=False)
    assert len(case.copy_pairs) == 4  # five sharers of the partial block: four forks, one in place
    kp, vp = oracle.copy_blocks(case.k_pool, case.v_pool, case.copy_pairs)
    kp, vp = oracle.paged_kv_write(kp, vp, case.k_new, case.v_new, case.slot_mapping)
    res = oracle.paged_prefill(case.q, case.query_start_loc, kp, vp, case.block_table,
                               case.context_lens, case.scale)
    qsl = case.query_start_loc.tolist()
    for b in range(5):
        k_l, v_l = case.extra["logical"][b]
        ref = oracle.causal_attention_contiguous(oracle.to_f64(case.q[qsl[b]:qsl[b + 1]]),
                                                 oracle.to_f64(k_l), oracle.to_f64(v_l), case.scale)
        for r in range(qsl[b + 1] - qsl[b]):
            assert np.array_equal(res[qsl[b] + r], ref[r])
    # the shared prefix rows are untouched by the forks: every table still reads the same prefix
    for b in range(5):
        assert np.array_equal(oracle.gather_history(kp, case.block_table[b], 44, 16),
                              oracle.to_f64(case.extra["logical"][0][0][:44]))


# ---------------------------------------------------------------------------------------------
# planted mistakes must fail a pin
# ---------------------------------------------------------------------------------------------

def _gqa_pin_fails():
    try:
        test_decode_matches_torch_sdpa(8, 2)
    except AssertionError:
        return True
    return False


def test_planted_wrong_gqa_map_is_caught(monkeypatch):
    monkeypatch.setattr(PO, "repeat_kv", lambda x, n: np.tile(x, (1, n, 1)))
    assert _gqa_pin_fails()


def test_planted_dropped_scale_is_caught(monkeypatch):
    real = PO.softmax_attention
    monkeypatch.setattr(PO, "softmax_attention", lambda q, k, v, scale: real(q, k, v, 1.0))
    assert _gqa_pin_fails()


def test_planted_causal_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(PO, "prefill_query_bound", lambda n, m, r: n - m + r)
    with pytest.raises(AssertionError):
        test_prefill_matches_torch_sdpa_with_offset_causal_mask()


def test_planted_slot_arithmetic_is_caught(monkeypatch):
    # offsets counted from the wrong end of each block
    monkeypatch.setattr(PO, "slot_of", lambda row, pos, S: int(row[pos // S]) * S + (S - 1 - pos % S))
    with pytest.raises(AssertionError):
        test_brute_force_tiny_workload_both_steps()


def test_sampled_rows_equal_full_decode():
    t = W.tiny_decode()
    full = oracle.paged_decode(t["q0"], t["k_pool"], t["v_pool"], t["block_table"], t["lens0"], t["scale"])
    rows = oracle.paged_decode_rows(t["q0"], t["k_pool"], t["v_pool"], t["block_table"], t["lens0"],
                                    t["scale"], [(0, 1), (1, 0)])
    assert np.array_equal(rows[(0, 1)], full[0, 4:8])
    assert np.array_equal(rows[(1, 0)], full[1, 0:4])


def test_transfer_blocks_between_pools():
    gen = torch.Generator().manual_seed(10)
    src_k = torch.randn((5, 4, 2, 8), generator=gen).to(torch.bfloat16)
    src_v = torch.randn((5, 4, 2, 8), generator=gen).to(torch.bfloat16)
    dst_k = torch.zeros((7, 4, 2, 8), dtype=torch.bfloat16)
    dst_v = torch.zeros((7, 4, 2, 8), dtype=torch.bfloat16)
    kd, vd = oracle.transfer_blocks(dst_k, dst_v, src_k, src_v, torch.tensor([[4, 0], [0, 6], [4, 3]]))
    assert torch.equal(kd[0], src_k[4]) and torch.equal(vd[6], src_v[0]) and torch.equal(kd[3], src_k[4])
    for blk in (1, 2, 4, 5):
        assert not kd[blk].float().abs().sum() and not vd[blk].float().abs().sum()
    assert not dst_k.float().abs().sum()  # inputs untouched
