"""Seeded synthetic inputs for the paged KV-cache path.

This module draws random numbers and lays them out as the paged cache expects them: K/V pools,
block tables, context lengths, slot mappings, queries and copy-on-write fork lists.  It holds none
of the attention arithmetic.  Both the GPU parity tests and the CPU oracle consume what it returns,
and `bench.py` uses it to build its device inputs.

Layout conventions (shared by every consumer, fixed here once):

* pools are ``[num_blocks, block_size, n_kv_heads, head_dim]`` — one pool for K, one for V
  (Pico-vLLM dev log #5, "core data structures and design": the device cache tensor is indexed
  block, token-in-block, kv head, head dim);
* a block table row lists the physical block id of each logical block of one sequence, int32,
  padded with -1 past the sequence's last block (Pico-vLLM dev log #5, ``get_block_table``);
* the slot of logical position ``j`` of a sequence is ``table[j // block_size] * block_size +
  j % block_size`` (JuliaPagedAttn README, "Block Layout": a physical block holds ``block_size``
  consecutive tokens), and ``slot_mapping`` is int64;
* ``context_lens`` counts the token(s) just written (Pico-vLLM dev log #5: the current token's K/V
  already exist in every layer, so lengths get the +1 correction).

Values are drawn in fp32 from a CPU ``torch.Generator`` and cast to the I/O dtype, so every machine
draws the same numbers.  Unused pool storage is filled with a sentinel (NaN for floating pools) so
that a stray read shows up as a NaN in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}

SEED_BASE = 1000  # seed of config c is SEED_BASE + c


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


# ----------------------------------------------------------------------------------------------
# building blocks
# ----------------------------------------------------------------------------------------------

def shuffled_block_tables(gen: torch.Generator, num_blocks: int, context_lens, block_size: int,
                          max_blocks_per_seq: int) -> torch.Tensor:
    """Give each sequence ``ceil(n_b / block_size)`` distinct physical ids, drawn without
    replacement from a shuffled ``arange(num_blocks)``; pad each row with -1."""
    perm = torch.randperm(num_blocks, generator=gen)
    batch = len(context_lens)
    table = torch.full((batch, max_blocks_per_seq), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(context_lens):
        nb = ceil_div(int(n), block_size)
        if nb > max_blocks_per_seq:
            raise ValueError("sequence needs more blocks than a table row holds")
        if pos + nb > num_blocks:
            raise ValueError("pool too small for the requested contexts")
        table[b, :nb] = perm[pos:pos + nb].to(torch.int32)
        pos += nb
    return table


def slots_for(table_row: torch.Tensor, positions, block_size: int) -> torch.Tensor:
    """int64 slot ids of the given logical positions of one sequence (layout convention above)."""
    pos = torch.as_tensor(positions, dtype=torch.int64)
    blk = table_row.to(torch.int64)[pos // block_size]
    if (blk < 0).any():
        raise ValueError("position beyond the sequence's allocated blocks")
    return blk * block_size + pos % block_size


def sentinel_pool(num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                  dtype: torch.dtype) -> torch.Tensor:
    return torch.full((num_blocks, block_size, n_kv_heads, head_dim), float("nan"), dtype=dtype)


def randn(gen: torch.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def fill_history(gen, k_pool, v_pool, table, lens, block_size, key_scale=None):
    """Write N(0,1) K and V values for logical positions ``0 .. n_b-1`` of every sequence.

    ``key_scale`` (optional, per sequence a float32 tensor of shape [n_b]) multiplies the keys of
    each position before the cast; it is how the long-context workload plants peaked rows."""
    Hkv, D = k_pool.shape[2], k_pool.shape[3]
    kf = k_pool.view(-1, Hkv, D)
    vf = v_pool.view(-1, Hkv, D)
    for b, n in enumerate(lens):
        n = int(n)
        if n == 0:
            continue
        s = slots_for(table[b], range(n), block_size)
        k = torch.randn((n, Hkv, D), generator=gen, dtype=torch.float32)
        v = torch.randn((n, Hkv, D), generator=gen, dtype=torch.float32)
        if key_scale is not None:
            k = k * key_scale[b].view(n, 1, 1)
        kf[s] = k.to(k_pool.dtype)
        vf[s] = v.to(v_pool.dtype)


@dataclass
class DecodeCase:
    """One decode step: write the new token of each sequence, then attend."""
    name: str
    dtype: torch.dtype
    block_size: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    scale: float
    k_pool: torch.Tensor          # [NB, S, Hkv, D]
    v_pool: torch.Tensor
    block_table: torch.Tensor     # int32 [B, max_blocks]
    context_lens: torch.Tensor    # int32 [B], counts the new token
    q: torch.Tensor               # [B, Hq, D]
    k_new: torch.Tensor           # [T, Hkv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor    # int64 [T]
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def num_blocks(self) -> int:
        return self.k_pool.shape[0]


def decode_case(name: str, seed: int, lens_before, *, n_q_heads: int, n_kv_heads: int, head_dim: int,
                block_size: int, dtype: torch.dtype, num_blocks: int, max_blocks_per_seq: int,
                key_outlier_frac: float = 0.0, key_outlier_scale: float = 1.0) -> DecodeCase:
    """A decode step over sequences whose history holds ``lens_before[b]`` tokens.

    The step writes one new token per sequence at position ``lens_before[b]`` and then attends
    over ``lens_before[b] + 1`` tokens.  Block tables already cover the new token's slot."""
    gen = _gen(seed)
    lens_after = [int(n) + 1 for n in lens_before]
    table = shuffled_block_tables(gen, num_blocks, lens_after, block_size, max_blocks_per_seq)
    k_pool = sentinel_pool(num_blocks, block_size, n_kv_heads, head_dim, dtype)
    v_pool = sentinel_pool(num_blocks, block_size, n_kv_heads, head_dim, dtype)
    key_scale = None
    if key_outlier_frac > 0.0:
        key_scale = []
        for n in lens_before:
            n = int(n)
            s = torch.ones(n, dtype=torch.float32)
            k = max(1, int(round(key_outlier_frac * n)))
            idx = torch.randperm(n, generator=gen)[:k]
            s[idx] = key_outlier_scale
            key_scale.append(s)
    fill_history(gen, k_pool, v_pool, table, lens_before, block_size, key_scale)
    B = len(lens_before)
    q = randn(gen, (B, n_q_heads, head_dim), dtype)
    k_new = randn(gen, (B, n_kv_heads, head_dim), dtype)
    v_new = randn(gen, (B, n_kv_heads, head_dim), dtype)
    slot = torch.cat([slots_for(table[b], [int(lens_before[b])], block_size) for b in range(B)])
    return DecodeCase(name=name, dtype=dtype, block_size=block_size, n_q_heads=n_q_heads,
                      n_kv_heads=n_kv_heads, head_dim=head_dim, scale=1.0 / math.sqrt(head_dim),
                      k_pool=k_pool, v_pool=v_pool, block_table=table,
                      context_lens=torch.tensor(lens_after, dtype=torch.int32), q=q,
                      k_new=k_new, v_new=v_new, slot_mapping=slot,
                      extra={"lens_before": [int(n) for n in lens_before]})


# ----------------------------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------------------------

def tiny_decode() -> dict:
    """Tiny decode: 2 sequences at 17 and 40 tokens, block_size 16, 8 query / 2 KV heads, head_dim
    64, fp32, a 16-block pool with a random permutation as the tables (partial last blocks).

    Returns the first step (attend over {17, 40}), then the write of one new token per sequence at
    positions 17 and 40 and the second step (attend over {18, 41}).  The tables already hold the
    block each new token lands in (positions 17 and 40 fall inside blocks 1 and 2)."""
    gen = _gen(SEED_BASE + 1)
    S, Hq, Hkv, D, NB = 16, 8, 2, 64, 16
    lens0 = [17, 40]
    lens1 = [18, 41]
    perm = torch.randperm(NB, generator=gen).to(torch.int32)
    table = torch.full((2, 3), -1, dtype=torch.int32)
    table[0, :2] = perm[0:2]
    table[1, :3] = perm[2:5]
    k_pool = sentinel_pool(NB, S, Hkv, D, torch.float32)
    v_pool = sentinel_pool(NB, S, Hkv, D, torch.float32)
    fill_history(gen, k_pool, v_pool, table, lens0, S)
    q0 = randn(gen, (2, Hq, D), torch.float32)
    k_new = randn(gen, (2, Hkv, D), torch.float32)
    v_new = randn(gen, (2, Hkv, D), torch.float32)
    q1 = randn(gen, (2, Hq, D), torch.float32)
    slot = torch.cat([slots_for(table[b], [lens0[b]], S) for b in range(2)])
    return dict(block_size=S, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, dtype=torch.float32,
                scale=1.0 / math.sqrt(D), k_pool=k_pool, v_pool=v_pool, block_table=table,
                lens0=torch.tensor(lens0, dtype=torch.int32), q0=q0, k_new=k_new, v_new=v_new,
                slot_mapping=slot, lens1=torch.tensor(lens1, dtype=torch.int32), q1=q1)


GPT2_BATCHES = (1, 2, 4, 8)
GPT2_CONTEXTS = (128, 256, 512, 1024, 2048)
GPT2_LAYERS = 12


def gpt2_decode(batch: int, context: int, layer: int = 0) -> DecodeCase:
    """GPT-2-small-shaped decode cell: 12 query = 12 KV heads, head_dim 64, block_size 16, fp16;
    every sequence at ``context`` tokens (the new one included); pool 1.25x the blocks needed,
    shuffled.  ``layer`` picks one of the 12 layers' independent pools."""
    S = 16
    need = batch * ceil_div(context, S)
    nb = ceil_div(5 * need, 4)
    seed = SEED_BASE + 2 + 7919 * (1 + GPT2_BATCHES.index(batch) * 5 + GPT2_CONTEXTS.index(context)) + 104729 * layer
    return decode_case(f"gpt2_b{batch}_n{context}_l{layer}", seed, [context - 1] * batch,
                       n_q_heads=12, n_kv_heads=12, head_dim=64, block_size=S, dtype=torch.float16,
                       num_blocks=nb, max_blocks_per_seq=ceil_div(context, S))


LLAMA_BATCH = 64
LLAMA_POOL = 40_000
LLAMA_MIN_CTX, LLAMA_MAX_CTX = 512, 4096


def llama_context_lens(seed: int = SEED_BASE + 3) -> list:
    """Context lengths (new token included) of the Llama-3-8B-shaped serving batch: uniform
    integers in [512, 4096]."""
    gen = _gen(seed)
    return [int(x) for x in torch.randint(LLAMA_MIN_CTX, LLAMA_MAX_CTX + 1, (LLAMA_BATCH,), generator=gen)]


def llama_decode(batch: int | None = None) -> DecodeCase:
    """Llama-3-8B-shaped serving decode: 32 query / 8 KV heads, head_dim 128, block_size 16, bf16;
    batch 64 with context lengths uniform in [512, 4096]; tables drawn without replacement from a
    shuffled 40,000-block pool; one new token per sequence written through slot_mapping."""
    lens = llama_context_lens()
    if batch is not None:
        lens = lens[:batch]
    return decode_case("llama3_8b_decode", SEED_BASE + 3, [n - 1 for n in lens], n_q_heads=32,
                       n_kv_heads=8, head_dim=128, block_size=16, dtype=torch.bfloat16,
                       num_blocks=LLAMA_POOL, max_blocks_per_seq=LLAMA_MAX_CTX // 16)


LONG_LENS = (32768, 65536, 98304, 131072)


def long_context_decode(lens=LONG_LENS) -> DecodeCase:
    """Long-context split-K decode: 32 query / 8 KV heads, head_dim 128, block_size 16, bf16; batch
    4 at 32K/64K/96K/128K tokens; 1% of each sequence's token positions have their keys scaled x8
    (peaked softmax rows); pool 1.25x the blocks needed, shuffled."""
    S = 16
    need = sum(ceil_div(n, S) for n in lens)
    return decode_case("long_context_decode", SEED_BASE + 4, [n - 1 for n in lens], n_q_heads=32,
                       n_kv_heads=8, head_dim=128, block_size=S, dtype=torch.bfloat16,
                       num_blocks=ceil_div(5 * need, 4), max_blocks_per_seq=ceil_div(max(lens), S),
                       key_outlier_frac=0.01, key_outlier_scale=8.0)


@dataclass
class PrefillCase:
    """Chunked prefill: write each sequence's new chunk, then attend causally over its history."""
    name: str
    dtype: torch.dtype
    block_size: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    scale: float
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor       # int32 [B, max_blocks] (after any copy-on-write fork)
    context_lens: torch.Tensor      # int32 [B], history + chunk
    query_start_loc: torch.Tensor   # int32 [B+1]
    q: torch.Tensor                 # [sum(m_b), Hq, D]
    k_new: torch.Tensor             # [T, Hkv, D] tokens written before the prefill
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # int64 [T]
    copy_pairs: torch.Tensor        # int64 [n, 2] (src, dst) forks to run before the write
    extra: dict = field(default_factory=dict)


def _prefix_shared_case(name, seed, *, batch, prefix, suffix_max, chunk, block_size, n_q_heads,
                        n_kv_heads, head_dim, dtype, num_blocks, suffix_in_cache: bool,
                        fixed_suffix=None) -> PrefillCase:
    """Sequences sharing a prefix, each with its own suffix and a new chunk.

    The prefix blocks are shared (one physical copy, refcount = batch).  With ``suffix_in_cache`` the
    suffix tokens already sit in the cache and only the chunk is written before the prefill;
    otherwise suffix and chunk are both written.  When the prefix ends inside a block, the first
    write of each sequence lands in that shared partial block: a host-side refcount decides a
    copy-on-write fork (allocate, copy, retarget the table entry, decrement), the last sharer
    writing in place (JuliaPagedAttn README, "Copy-on-Write").  ``extra['logical']`` keeps every
    sequence's unshared history values (the copy the oracle reads)."""
    gen = _gen(seed)
    S = block_size
    if suffix_in_cache and prefix % S != 0:
        raise ValueError("a suffix already in the cache cannot follow a shared partial block")
    if fixed_suffix is None:
        suffix = [int(x) for x in torch.randint(0, suffix_max + 1, (batch,), generator=gen)]
    else:
        suffix = list(fixed_suffix)
    lens = [prefix + s + chunk for s in suffix]
    max_blocks = ceil_div(prefix + suffix_max + chunk, S)
    perm = [int(x) for x in torch.randperm(num_blocks, generator=gen)]
    free = list(perm)
    n_prefix_blocks = ceil_div(prefix, S)
    prefix_ids = [free.pop() for _ in range(n_prefix_blocks)]
    refcount = {pid: batch for pid in prefix_ids}
    table = torch.full((batch, max_blocks), -1, dtype=torch.int32)
    for b in range(batch):
        table[b, :n_prefix_blocks] = torch.tensor(prefix_ids, dtype=torch.int32)
    k_pool = sentinel_pool(num_blocks, S, n_kv_heads, head_dim, dtype)
    v_pool = sentinel_pool(num_blocks, S, n_kv_heads, head_dim, dtype)
    # shared prefix values (one copy in the pool)
    kp = randn(gen, (prefix, n_kv_heads, head_dim), dtype)
    vp = randn(gen, (prefix, n_kv_heads, head_dim), dtype)
    kf = k_pool.view(-1, n_kv_heads, head_dim)
    vf = v_pool.view(-1, n_kv_heads, head_dim)
    s0 = slots_for(table[0], range(prefix), S)
    kf[s0] = kp
    vf[s0] = vp
    # per-sequence private blocks for the rest of the context
    for b in range(batch):
        for lb in range(n_prefix_blocks, ceil_div(lens[b], S)):
            table[b, lb] = free.pop()
    # values of every sequence's suffix and chunk
    ks = [randn(gen, (suffix[b], n_kv_heads, head_dim), dtype) for b in range(batch)]
    vs = [randn(gen, (suffix[b], n_kv_heads, head_dim), dtype) for b in range(batch)]
    kc = [randn(gen, (chunk, n_kv_heads, head_dim), dtype) for b in range(batch)]
    vc = [randn(gen, (chunk, n_kv_heads, head_dim), dtype) for b in range(batch)]
    q = randn(gen, (batch * chunk, n_q_heads, head_dim), dtype)
    copy_pairs = []
    k_w, v_w, slot_w = [], [], []
    partial = prefix % S != 0
    for b in range(batch):
        first_write = prefix if not suffix_in_cache else prefix + suffix[b]
        lb = first_write // S
        if partial and lb == n_prefix_blocks - 1:
            shared = int(table[b, lb])
            if refcount[shared] > 1:
                new = free.pop()
                copy_pairs.append((shared, new))
                table[b, lb] = new
                refcount[shared] -= 1
        if suffix_in_cache:
            sl = slots_for(table[b], range(prefix, prefix + suffix[b]), S)
            kf[sl] = ks[b]
            vf[sl] = vs[b]
        else:
            k_w.append(ks[b]); v_w.append(vs[b])
            slot_w.append(slots_for(table[b], range(prefix, prefix + suffix[b]), S))
        k_w.append(kc[b]); v_w.append(vc[b])
        slot_w.append(slots_for(table[b], range(prefix + suffix[b], lens[b]), S))
    qsl = torch.tensor([b * chunk for b in range(batch + 1)], dtype=torch.int32)
    logical = [(torch.cat([kp, ks[b], kc[b]]), torch.cat([vp, vs[b], vc[b]])) for b in range(batch)]
    return PrefillCase(
        name=name, dtype=dtype, block_size=S, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
        head_dim=head_dim, scale=1.0 / math.sqrt(head_dim), k_pool=k_pool, v_pool=v_pool,
        block_table=table, context_lens=torch.tensor(lens, dtype=torch.int32),
        query_start_loc=qsl, q=q, k_new=torch.cat(k_w), v_new=torch.cat(v_w),
        slot_mapping=torch.cat(slot_w), copy_pairs=torch.tensor(copy_pairs, dtype=torch.int64).view(-1, 2),
        extra={"suffix": suffix, "prefix": prefix, "chunk": chunk, "logical": logical,
               "prefix_blocks": prefix_ids})


PREFILL_BATCH = 128
PREFILL_PREFIX = 1024
PREFILL_COW_PREFIX = 1000
PREFILL_SUFFIX_MAX = 512
PREFILL_CHUNK = 256
PREFILL_POOL = 4096


def prefill_cow(batch: int = PREFILL_BATCH, cow_arm: bool = False) -> PrefillCase:
    """Chunked prefill with a shared prefix: 32 query / 8 KV heads, head_dim 128, block_size 32,
    bf16; 128 sequences share a 1024-token prefix (32 blocks with refcount 128), each with its own
    suffix of uniform length in [0, 512] already in the cache and a causal chunk of 256 new tokens
    written and then prefilled; pool of 4096 blocks.

    ``cow_arm`` shortens the shared prefix to 1000 tokens so that block 31 is a shared partial
    block: each sequence's first write (its suffix, written in this arm) lands there and forks it."""
    if cow_arm:
        return _prefix_shared_case("prefill_cow_fork", SEED_BASE + 5 + 100, batch=batch,
                                   prefix=PREFILL_COW_PREFIX, suffix_max=PREFILL_SUFFIX_MAX,
                                   chunk=PREFILL_CHUNK, block_size=32, n_q_heads=32, n_kv_heads=8,
                                   head_dim=128, dtype=torch.bfloat16, num_blocks=PREFILL_POOL,
                                   suffix_in_cache=False)
    return _prefix_shared_case("prefill_shared_prefix", SEED_BASE + 5, batch=batch,
                               prefix=PREFILL_PREFIX, suffix_max=PREFILL_SUFFIX_MAX,
                               chunk=PREFILL_CHUNK, block_size=32, n_q_heads=32, n_kv_heads=8,
                               head_dim=128, dtype=torch.bfloat16, num_blocks=PREFILL_POOL,
                               suffix_in_cache=True)


def small_prefill(seed: int, *, batch: int, prefix: int, suffix_max: int, chunk: int, block_size: int,
                  n_q_heads: int, n_kv_heads: int, head_dim: int, dtype: torch.dtype,
                  num_blocks: int, suffix_in_cache: bool = True, fixed_suffix=None) -> PrefillCase:
    """Reduced prefill cases for fast parity tests (same recipe, smaller sizes)."""
    return _prefix_shared_case(f"prefill_small_{seed}", seed, batch=batch, prefix=prefix,
                               suffix_max=suffix_max, chunk=chunk, block_size=block_size,
                               n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                               dtype=dtype, num_blocks=num_blocks, suffix_in_cache=suffix_in_cache,
                               fixed_suffix=fixed_suffix)


def varlen_prefill(seed: int, *, hist_lens, chunk_lens, block_size: int, n_q_heads: int,
                   n_kv_heads: int, head_dim: int, dtype: torch.dtype, num_blocks: int) -> PrefillCase:
    """Prefill with ragged chunk lengths (including empty chunks) over private histories."""
    gen = _gen(seed)
    S = block_size
    lens = [int(h) + int(c) for h, c in zip(hist_lens, chunk_lens)]
    max_blocks = max(1, max(ceil_div(n, S) for n in lens))
    table = shuffled_block_tables(gen, num_blocks, lens, S, max_blocks)
    k_pool = sentinel_pool(num_blocks, S, n_kv_heads, head_dim, dtype)
    v_pool = sentinel_pool(num_blocks, S, n_kv_heads, head_dim, dtype)
    fill_history(gen, k_pool, v_pool, table, hist_lens, S)
    B = len(lens)
    total = sum(int(c) for c in chunk_lens)
    q = randn(gen, (total, n_q_heads, head_dim), dtype)
    k_new = randn(gen, (total, n_kv_heads, head_dim), dtype)
    v_new = randn(gen, (total, n_kv_heads, head_dim), dtype)
    slots = [slots_for(table[b], range(int(hist_lens[b]), lens[b]), S) for b in range(B)]
    qsl = [0]
    for c in chunk_lens:
        qsl.append(qsl[-1] + int(c))
    return PrefillCase(
        name=f"prefill_varlen_{seed}", dtype=dtype, block_size=S, n_q_heads=n_q_heads,
        n_kv_heads=n_kv_heads, head_dim=head_dim, scale=1.0 / math.sqrt(head_dim), k_pool=k_pool,
        v_pool=v_pool, block_table=table, context_lens=torch.tensor(lens, dtype=torch.int32),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32), q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64),
        copy_pairs=torch.zeros((0, 2), dtype=torch.int64), extra={})


# ----------------------------------------------------------------------------------------------
# device-resident inputs for timing (values only need to be finite and seeded)
# ----------------------------------------------------------------------------------------------

def device_decode_inputs(lens, *, n_q_heads, n_kv_heads, head_dim, block_size, dtype, num_blocks,
                         max_blocks_per_seq, device, seed, layers: int = 1):
    """Device tensors for timing a decode step: ``layers`` independent K/V pools (so consecutive
    timed steps touch different memory), tables and slot mappings built on the host, values drawn
    on the device from a seeded generator."""
    gen = _gen(seed)
    table = shuffled_block_tables(gen, num_blocks, lens, block_size, max_blocks_per_seq)
    slot = torch.cat([slots_for(table[b], [int(lens[b]) - 1], block_size) for b in range(len(lens))])
    dgen = torch.Generator(device=device)
    dgen.manual_seed(seed)
    pools = []
    for _ in range(layers):
        kp = torch.randn((num_blocks, block_size, n_kv_heads, head_dim), generator=dgen, device=device,
                         dtype=torch.float32).to(dtype)
        vp = torch.randn((num_blocks, block_size, n_kv_heads, head_dim), generator=dgen, device=device,
                         dtype=torch.float32).to(dtype)
        pools.append((kp, vp))
    B = len(lens)
    q = torch.randn((B, n_q_heads, head_dim), generator=gen, dtype=torch.float32).to(dtype)
    k_new = torch.randn((B, n_kv_heads, head_dim), generator=gen, dtype=torch.float32).to(dtype)
    v_new = torch.randn((B, n_kv_heads, head_dim), generator=gen, dtype=torch.float32).to(dtype)
    return dict(pools=pools, block_table=table, slot_mapping=slot,
                context_lens=torch.tensor([int(n) for n in lens], dtype=torch.int32),
                q=q, k_new=k_new, v_new=v_new)
