"""CPU oracle for paged KV-cache attention.  TEST INFRASTRUCTURE ONLY.

This module is the slow, plainly-correct definition that the CUDA library is checked against.  Only
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it; the
library never does, and this module imports nothing from the library.

Every floating-point result is computed in float64 from the values actually stored in the caller's
tensors (a bf16/fp16 pool is upcast exactly).  Pools and tables may be torch CPU tensors or numpy
arrays; the bit-copy operations (the K/V write and the block copy) work on torch tensors of any
dtype and copy raw values.

Sources (page title, section):

* JuliaPagedAttn README, "Block Layout": a physical block holds the K and V of ``block_size``
  consecutive tokens for every KV head; "Architecture": attention reaches the cache through a
  block-table indirection.
* Pico-vLLM dev log #5 "Paged Attention", "core data structures and design": the device cache is
  ``[num_blocks, block_size, num_kv_heads, head_dim]`` per layer and per K/V; ``get_block_table``
  returns the int32 physical ids of a sequence's logical blocks; the sequence length gets the +1
  correction because the current token's K/V already exist when a layer attends.
* JuliaPagedAttn README, "Online Softmax": single pass with running maximum, running sum and an
  accumulator rescaled by the correction; output = accumulator / running sum.
* nanoserve "Day 19: the fused paged read wired into attention", "Why it matters": the read through
  the block table must equal gathering the scattered blocks into one contiguous history and running
  ordinary attention over it; "What I learned" item 4: the cache stores the compact KV heads and the
  GQA repeat happens at read time; "What I added today": ``n_rep`` and ``scale=None`` arguments.
* JuliaPagedAttn README, "Copy-on-Write": a write into a shared block allocates a new block, copies
  the data, updates the table and decrements the refcount.
* JuliaPagedAttn README, "Features": batched prefill processes all prompt positions in one call.

Readings where the pages are silent (each also listed in the design notes):

* query head ``i`` reads KV head ``i // (Hq // Hkv)`` (contiguous groups, as a repeat along the head
  axis produces);
* the query of a decode step attends to every one of the ``context_lens[b]`` tokens, itself included;
* a prefill chunk of ``m`` queries occupies the last ``m`` positions of the context; query ``r``
  (0-based) attends to positions ``0 .. n_b - m + r`` inclusive;
* an empty context yields a zero output;
* a negative slot in ``slot_mapping`` means "no write" for that token;
* a split-K partition that holds no token contributes nothing to the merge.
"""
from __future__ import annotations

import numpy as np

try:  # torch is optional for the numeric parts; used only to accept torch tensors
    import torch
except Exception:  # pragma: no cover
    torch = None


# ----------------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------------

def _is_torch(x) -> bool:
    return torch is not None and isinstance(x, torch.Tensor)


def to_f64(x) -> np.ndarray:
    """Exact upcast of stored values to a float64 numpy array."""
    if _is_torch(x):
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def to_int(x) -> np.ndarray:
    if _is_torch(x):
        return x.detach().to("cpu").to(torch.int64).numpy()
    return np.asarray(x, dtype=np.int64)


# ----------------------------------------------------------------------------------------------
# block-table addressing and the contiguous gather
# ----------------------------------------------------------------------------------------------

def slot_of(table_row, pos: int, block_size: int) -> int:
    """Physical slot of logical position ``pos``: block ``table_row[pos // block_size]``, token
    ``pos % block_size`` inside it (JuliaPagedAttn "Block Layout"; Pico-vLLM ``get_block_table``)."""
    return int(table_row[pos // block_size]) * block_size + pos % block_size


def history_slots(table_row, n: int, block_size: int) -> list:
    return [slot_of(table_row, j, block_size) for j in range(n)]


def gather_history(pool, table_row, n: int, block_size: int, kv_head=None) -> np.ndarray:
    """The contiguous ``[n, Hkv, D]`` float64 history of one sequence, read through its block table
    (nanoserve Day 19 "Why it matters": the gather path).  With ``kv_head`` set, only that head is
    gathered and the result is ``[n, 1, D]``."""
    NB, S, Hkv, D = pool.shape
    assert S == block_size
    slots = history_slots(to_int(table_row), n, block_size)
    heads = slice(None) if kv_head is None else slice(kv_head, kv_head + 1)
    if n == 0:
        return np.zeros((0, Hkv if kv_head is None else 1, D))
    if _is_torch(pool):
        flat = pool.reshape(NB * S, Hkv, D)
        rows = flat[torch.as_tensor(slots, dtype=torch.int64)][:, heads]
        return rows.to(torch.float64).numpy()
    flat = np.asarray(pool).reshape(NB * S, Hkv, D)
    return flat[slots][:, heads].astype(np.float64)


def repeat_kv(x: np.ndarray, n_rep: int) -> np.ndarray:
    """``[n, Hkv, D] -> [n, Hkv * n_rep, D]``: query head ``i`` sees KV head ``i // n_rep``
    (nanoserve Day 19 "What I learned" item 4: the repeat happens on the read side)."""
    return np.repeat(x, n_rep, axis=1)


# ----------------------------------------------------------------------------------------------
# attention over a contiguous history
# ----------------------------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Two-pass softmax attention of ``q [H, D]`` over ``k, v [n, H, D]`` (heads already repeated).

    ``z[h, j] = scale * <q[h], k[j, h]>``, ``p = exp(z - max_j z) / sum_j exp(z - max_j z)``,
    ``out[h] = sum_j p[h, j] v[j, h]``.  An empty history gives zeros."""
    H, D = q.shape
    n = k.shape[0]
    if n == 0:
        return np.zeros((H, D))
    z = scale * np.einsum("hd,jhd->hj", q, k)
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    p = e / e.sum(axis=1, keepdims=True)
    return np.einsum("hj,jhd->hd", p, v)


def online_softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Single-pass attention in the order of JuliaPagedAttn "Online Softmax": one token at a time,
    keep a running maximum, a running sum and an accumulator, rescale both by ``exp(old_max -
    new_max)`` when the maximum grows, and divide at the end."""
    H, D = q.shape
    out = np.zeros((H, D))
    for h in range(H):
        running_max = -np.inf
        running_sum = 0.0
        acc = np.zeros(D)
        for t in range(k.shape[0]):
            score = float(np.dot(q[h], k[t, h])) * scale
            new_max = max(running_max, score)
            correction = np.exp(running_max - new_max) if running_max != -np.inf else 0.0
            weight = np.exp(score - new_max)
            running_sum = running_sum * correction + weight
            acc = acc * correction + weight * v[t, h]
            running_max = new_max
        out[h] = acc / running_sum if running_sum > 0.0 else 0.0
    return out


# ----------------------------------------------------------------------------------------------
# split-K partials and the log-sum-exp merge
# ----------------------------------------------------------------------------------------------

def partition_partials(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, bounds) -> list:
    """Per token range ``[lo, hi)`` of ``bounds``: ``(m, l, acc)`` with ``m[h] = max_j z[h, j]``,
    ``l[h] = sum_j exp(z[h, j] - m[h])`` and ``acc[h] = sum_j exp(z[h, j] - m[h]) v[j, h]``
    (unnormalised).  An empty range gives ``m = -inf, l = 0, acc = 0``."""
    H, D = q.shape
    parts = []
    for lo, hi in bounds:
        if hi <= lo:
            parts.append((np.full(H, -np.inf), np.zeros(H), np.zeros((H, D))))
            continue
        z = scale * np.einsum("hd,jhd->hj", q, k[lo:hi])
        m = z.max(axis=1)
        e = np.exp(z - m[:, None])
        parts.append((m, e.sum(axis=1), np.einsum("hj,jhd->hd", e, v[lo:hi])))
    return parts


def lse_merge(parts) -> np.ndarray:
    """Exact merge of partition partials: ``M = max_p m_p``, ``L = sum_p l_p exp(m_p - M)``,
    ``out = sum_p acc_p exp(m_p - M) / L``; partitions with ``l_p = 0`` are skipped."""
    H, D = parts[0][2].shape
    out = np.zeros((H, D))
    for h in range(H):
        live = [(m[h], l[h], a[h]) for m, l, a in parts if l[h] > 0.0]
        if not live:
            continue
        M = max(m for m, _, _ in live)
        L = sum(l * np.exp(m - M) for m, l, _ in live)
        out[h] = sum(a * np.exp(m - M) for m, _, a in live) / L
    return out


# ----------------------------------------------------------------------------------------------
# the paged operations
# ----------------------------------------------------------------------------------------------

def paged_decode(q, k_pool, v_pool, block_table, context_lens, scale: float) -> np.ndarray:
    """Decode attention through the block table.

    For each sequence ``b``: gather its ``context_lens[b]`` tokens of K and V contiguously, repeat the
    KV heads up to the query heads, and run two-pass softmax attention.  Returns ``[B, Hq, D]``
    float64."""
    qf = to_f64(q)
    B, Hq, D = qf.shape
    S, Hkv = k_pool.shape[1], k_pool.shape[2]
    assert Hq % Hkv == 0
    g = Hq // Hkv
    table = to_int(block_table)
    lens = to_int(context_lens)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(lens[b])
        kc = repeat_kv(gather_history(k_pool, table[b], n, S), g)
        vc = repeat_kv(gather_history(v_pool, table[b], n, S), g)
        out[b] = softmax_attention(qf[b], kc, vc, scale)
    return out


def paged_decode_rows(q, k_pool, v_pool, block_table, context_lens, scale: float, rows) -> dict:
    """``paged_decode`` restricted to sampled ``(b, kv_head)`` rows, for full-size cases.
    Returns ``{(b, kv_head): [g, D] float64}``."""
    qf = to_f64(q)
    B, Hq, D = qf.shape
    S, Hkv = k_pool.shape[1], k_pool.shape[2]
    g = Hq // Hkv
    table = to_int(block_table)
    lens = to_int(context_lens)
    res = {}
    for b, kvh in rows:
        n = int(lens[b])
        kc = gather_history(k_pool, table[b], n, S, kv_head=kvh)
        vc = gather_history(v_pool, table[b], n, S, kv_head=kvh)
        res[(b, kvh)] = softmax_attention(qf[b, kvh * g:(kvh + 1) * g], repeat_kv(kc, g),
                                          repeat_kv(vc, g), scale)
    return res


def prefill_query_bound(n_b: int, m: int, r: int) -> int:
    """Number of keys query ``r`` of an ``m``-query chunk sees in a context of ``n_b`` tokens: the
    chunk fills the last ``m`` positions and attention is causal and includes the query itself."""
    return n_b - m + r + 1


def paged_prefill(q, query_start_loc, k_pool, v_pool, block_table, context_lens, scale: float,
                  seqs=None, queries=None) -> dict:
    """Causal chunked prefill through the block table.

    Sequence ``b`` owns queries ``query_start_loc[b] .. query_start_loc[b+1]-1``.  Query ``r`` of the
    chunk attends over positions ``0 .. n_b - m + r`` of the gathered history (causal mask applied
    by slicing the history, not by adding ``-inf``).  Returns ``{token_index: [Hq, D]}`` for the
    selected sequences (all if ``seqs`` is None) and, per sequence, the selected chunk rows
    (``queries`` = list of r, or None for all)."""
    qf_all = q
    qsl = to_int(query_start_loc)
    lens = to_int(context_lens)
    table = to_int(block_table)
    S, Hkv = k_pool.shape[1], k_pool.shape[2]
    Hq = q.shape[1]
    g = Hq // Hkv
    B = len(lens)
    res = {}
    for b in (range(B) if seqs is None else seqs):
        lo, hi = int(qsl[b]), int(qsl[b + 1])
        m = hi - lo
        if m == 0:
            continue
        n = int(lens[b])
        kc = repeat_kv(gather_history(k_pool, table[b], n, S), g)
        vc = repeat_kv(gather_history(v_pool, table[b], n, S), g)
        for r in (range(m) if queries is None else [r for r in queries if r < m]):
            t = lo + r
            nk = prefill_query_bound(n, m, r)
            res[t] = softmax_attention(to_f64(qf_all[t]), kc[:nk], vc[:nk], scale)
    return res


def causal_attention_contiguous(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Causal attention of an ``m``-query chunk that ends a contiguous ``n``-token history:
    ``q [m, Hq, D]``, ``k, v [n, Hkv, D]`` (compact heads) -> ``[m, Hq, D]``."""
    m, Hq, D = q.shape
    n, Hkv, _ = k.shape
    g = Hq // Hkv
    kr, vr = repeat_kv(k, g), repeat_kv(v, g)
    out = np.zeros((m, Hq, D))
    for r in range(m):
        nk = prefill_query_bound(n, m, r)
        out[r] = softmax_attention(q[r], kr[:nk], vr[:nk], scale)
    return out


def paged_kv_write(k_pool, v_pool, k_new, v_new, slot_mapping):
    """Scatter this step's K/V into pool slots, one token after another: token ``t`` with slot
    ``s >= 0`` overwrites row ``s`` of ``pool.view(num_blocks * block_size, Hkv, D)`` with an exact
    bit copy; ``s < 0`` writes nothing.  Returns new (K, V) pools; the inputs are left untouched
    (nanoserve Day 19 "What I learned" item 2: the shared write scatters the K/V to this step's
    slots)."""
    kp, vp = k_pool.clone(), v_pool.clone()
    NB, S, Hkv, D = kp.shape
    kf, vf = kp.view(NB * S, Hkv, D), vp.view(NB * S, Hkv, D)
    slots = to_int(slot_mapping)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        kf[int(s)] = k_new[t]
        vf[int(s)] = v_new[t]
    return kp, vp


def copy_blocks(k_pool, v_pool, pairs):
    """For each ``(src, dst)`` pair in order, make physical block ``dst`` a bit copy of block
    ``src`` in both pools (the copy step of JuliaPagedAttn "Copy-on-Write").  Returns new pools."""
    kp, vp = k_pool.clone(), v_pool.clone()
    for src, dst in to_int(pairs).reshape(-1, 2):
        kp[int(dst)] = kp[int(src)]
        vp[int(dst)] = vp[int(src)]
    return kp, vp


def transfer_blocks(dst_k, dst_v, src_k, src_v, pairs):
    """Block swap between two pools (Pico-vLLM dev log #5 "Paged Attention", swap_out / swap_in): for
    each ``(src, dst)`` pair, block ``dst`` of the destination pools becomes a bit copy of block
    ``src`` of the source pools.  Returns new destination pools."""
    kd, vd = dst_k.clone(), dst_v.clone()
    for src, dst in to_int(pairs).reshape(-1, 2):
        kd[int(dst)] = src_k[int(src)]
        vd[int(dst)] = src_v[int(src)]
    return kd, vd
