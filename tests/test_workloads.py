"""Host-side checks of the seeded input generators (shapes, ranges, table validity)."""
import torch

import workloads as W


def test_tiny_workload_shape_and_partial_blocks():
    t = W.tiny_decode()
    assert t["k_pool"].shape == (16, 16, 2, 64) and t["k_pool"].dtype == torch.float32
    tab = t["block_table"]
    ids = [int(x) for x in tab.flatten() if x >= 0]
    assert len(ids) == 5 and len(set(ids)) == 5 and all(0 <= i < 16 for i in ids)
    assert t["lens0"].tolist() == [17, 40] and t["lens1"].tolist() == [18, 41]
    # new tokens land inside already-allocated blocks: logical 1 offset 1, logical 2 offset 8
    assert int(t["slot_mapping"][0]) == int(tab[0, 1]) * 16 + 1
    assert int(t["slot_mapping"][1]) == int(tab[1, 2]) * 16 + 8


def test_llama_lens_and_tables():
    lens = W.llama_context_lens()
    assert len(lens) == 64 and min(lens) >= 512 and max(lens) <= 4096
    assert any(n % 16 for n in lens)  # partial last blocks occur
    gen = torch.Generator().manual_seed(0)
    tab = W.shuffled_block_tables(gen, 40000, lens, 16, 256)
    used = tab[tab >= 0]
    assert used.numel() == sum(W.ceil_div(n, 16) for n in lens)
    assert torch.unique(used).numel() == used.numel()


def test_cow_arm_forks_every_sharer_but_the_last():
    c = W.small_prefill(3, batch=4, prefix=20, suffix_max=5, chunk=4, block_size=8, n_q_heads=2,
                        n_kv_heads=1, head_dim=8, dtype=torch.float32, num_blocks=32,
                        suffix_in_cache=False)
    assert c.copy_pairs.shape == (3, 2)
    shared = c.extra["prefix_blocks"][-1]
    assert all(int(s) == shared for s in c.copy_pairs[:, 0])
    assert sum(int(c.block_table[b, 2]) == shared for b in range(4)) == 1
    # every written slot is distinct
    assert torch.unique(c.slot_mapping).numel() == c.slot_mapping.numel()
