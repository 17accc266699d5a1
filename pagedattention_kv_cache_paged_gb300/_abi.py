"""ctypes binding of libpagedattn.so: argument marshalling only.

Every function here checks tensor shapes, dtypes, devices and contiguity, turns torch tensors into
raw device pointers and calls the C entry point of the same name on the current CUDA stream.  All
arithmetic runs in the library's CUDA kernels; there is no CPU or PyTorch fallback — if the shared
library is missing or fails to load, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedattn.so")

PA_BF16, PA_FP16, PA_FP32 = 0, 1, 2
_DTYPE_CODES = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16, torch.float32: PA_FP32}

PA_OK, PA_EINVAL, PA_EDTYPE, PA_ERANGE, PA_EWORKSPACE, PA_ECUDA, PA_EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
PA_OPT_CHECKED = 1
PA_DEVERR_BLOCK_ID, PA_DEVERR_SLOT, PA_DEVERR_CONTEXT_LEN = 1, 2, 4
PA_DEVERR_COPY_PAIR, PA_DEVERR_QUERY_LOC, PA_DEVERR_TIMEOUT = 8, 16, 32

_vp, _i64, _i32, _sz, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_float


class PaOpts(ctypes.Structure):
    """struct pa_opts of include/pagedattn.h: the per-call options of the ``_ex`` entry points."""
    _fields_ = [("kv_block_stride_bytes", ctypes.c_int64), ("decode_kernel", ctypes.c_int32),
                ("prefill_kernel", ctypes.c_int32), ("partition_tokens", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_opts_p = ctypes.POINTER(PaOpts)

# name -> (restype, argtypes), mirroring include/pagedattn.h
_KV_WRITE = [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _i32]
_DECODE = [_vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _i64, _i32, _f32, _i32, _i32, _i32, _i32, _vp, _sz]
_FUSED = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _i64, _i32, _f32, _i32, _i32, _i32, _i32, _vp, _sz]
_WS = [_i32, _i64, _i32, _i32, _i32, _i32]
_PREFILL = [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp, _i32, _i64, _i32, _f32, _i32, _i32, _i32, _i32]
_COPY = [_vp, _vp, _vp, _i64, _i64, _i64]
_SWAP = [_vp, _vp, _i64, _vp, _vp, _i64, _vp, _i64, _i64]
SIGNATURES = {
    "paged_kv_write": (_i32, _KV_WRITE + [_vp]),
    "paged_kv_write_ex": (_i32, _KV_WRITE + [_opts_p, _vp]),
    "paged_attention_decode": (_i32, _DECODE + [_vp]),
    "paged_attention_decode_ex": (_i32, _DECODE + [_opts_p, _vp]),
    "paged_attention_decode_workspace_size": (_sz, _WS),
    "paged_attention_decode_workspace_size_ex": (_sz, _WS + [_opts_p]),
    "pa_decode_split_plan": (_i32, _WS + [_i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32),
                                          ctypes.POINTER(_sz)]),
    "paged_attention_decode_fused": (_i32, _FUSED + [_vp]),
    "paged_attention_decode_fused_ex": (_i32, _FUSED + [_opts_p, _vp]),
    "paged_attention_prefill": (_i32, _PREFILL + [_vp]),
    "paged_attention_prefill_ex": (_i32, _PREFILL + [_opts_p, _vp]),
    "copy_blocks": (_i32, _COPY + [_vp]),
    "copy_blocks_ex": (_i32, _COPY + [_opts_p, _vp]),
    "swap_blocks": (_i32, _SWAP + [_vp]),
    "swap_blocks_ex": (_i32, _SWAP + [_opts_p, _vp]),
    "paged_attention_lse_merge": (_i32, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp]),
    "paged_attention_decode_static_scratch": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _i64, _i32, _f32,
                                                     _i32, _i32, _i32, _i32, _vp]),
    "pa_set_checked_mode": (_i32, [_i32]),
    "pa_set_option": (_i32, [_i32, _i64]),
    "pa_get_option": (_i64, [_i32]),
    "pa_last_cuda_error": (_i32, []),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_device_error_flags": (_i32, [_i32, _vp]),
    "pa_selftest_bounded_wait": (_i32, [_i64, _vp, _vp]),
    "pa_launch_count": (ctypes.c_uint64, []),
    "pa_version": (ctypes.c_char_p, []),
}

_lib = None
_lock = threading.Lock()


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn} failed with status {status} ({detail})")


def load_library(path: str | None = None):
    """Load libpagedattn.so (built in-tree by build.py) and bind its signatures.  Raises if missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or os.environ.get("PAGEDATTN_LIB", LIB_PATH)
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m pagedattention_kv_cache_paged_gb300.build` "
                               "(the library has no CPU fallback)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != PA_OK:
        lib = load_library()
        detail = lib.pa_status_string(status).decode()
        if status == PA_ECUDA:
            detail += f", cudaError {lib.pa_last_cuda_error()}"
        raise PagedAttnError(fn, status, detail)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None, contiguous: bool = True) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _code(dtype: torch.dtype) -> int:
    if dtype not in _DTYPE_CODES:
        raise TypeError(f"unsupported dtype {dtype}")
    return _DTYPE_CODES[dtype]


def _pool_dims(k_pool: torch.Tensor, v_pool: torch.Tensor):
    if k_pool.dim() != 4 or k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype:
        raise ValueError("k_pool and v_pool must both be [num_blocks, block_size, n_kv_heads, head_dim] of one dtype")
    return tuple(int(x) for x in k_pool.shape)


def unified_views(pool: torch.Tensor):
    """K and V views ``[num_blocks, block_size, n_kv_heads, head_dim]`` of a unified K/V pool
    ``[num_blocks, 2, block_size, n_kv_heads, head_dim]`` (block b holds its keys, then its values).
    Every call accepts them as ``k_pool, v_pool``: their block stride (twice a block) travels with
    the call."""
    if pool.dim() != 5 or pool.shape[1] != 2 or not pool.is_contiguous():
        raise ValueError("a unified pool is a contiguous [num_blocks, 2, block_size, n_kv_heads, head_dim] tensor")
    return pool[:, 0], pool[:, 1]


def _pool(t: torch.Tensor, name: str, dtype=None, host_ok: bool = False) -> int:
    """Pointer of a K or V pool after checking its layout: each block [block_size, n_kv_heads,
    head_dim] contiguous, blocks any multiple of 16 bytes apart (at least one block)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 4:
        raise ValueError(f"{name} must be [num_blocks, block_size, n_kv_heads, head_dim]")
    NB, S, Hkv, D = (int(x) for x in t.shape)
    st = tuple(t.stride())
    if st[1:] != (Hkv * D, D, 1) or (NB > 1 and st[0] < S * Hkv * D) or (st[0] * t.element_size()) % 16:
        raise ValueError(f"{name}: each block must be contiguous and blocks at least one block and a multiple of "
                         f"16 bytes apart (strides {tuple(st)})")
    return t.data_ptr()


def _block_stride_bytes(k_pool: torch.Tensor, v_pool: torch.Tensor) -> int:
    """kv_block_stride_bytes of a call: 0 for contiguous pools, else the pools' common block stride."""
    NB, S, Hkv, D = (int(x) for x in k_pool.shape)
    ks, vs = int(k_pool.stride(0)), int(v_pool.stride(0))
    if NB <= 1:
        return 0
    if ks != vs:
        raise ValueError(f"k_pool and v_pool must share one block stride (got {ks} and {vs} elements)")
    return 0 if ks == S * Hkv * D else ks * k_pool.element_size()


def make_opts(kv_block_stride_bytes: int = 0, decode_kernel: int = 0, prefill_kernel: int = 0,
              partition_tokens: int = 0) -> PaOpts:
    """A pa_opts for the ``_ex`` entry points (decode_kernel: 0 auto, 1 CUDA cores, 2 tensor cores;
    prefill_kernel: 0 auto, 1 CUDA cores, 2 tcgen05; partition_tokens: 0 automatic)."""
    return PaOpts(int(kv_block_stride_bytes), int(decode_kernel), int(prefill_kernel), int(partition_tokens), 0)


# ----------------------------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------------------------

def paged_kv_write(k_new, v_new, slot_mapping, k_pool, v_pool, stream=None):
    """Scatter ``k_new, v_new [T, Hkv, D]`` into the pools at ``slot_mapping`` (int64 [T])."""
    lib = load_library()
    NB, S, Hkv, D = _pool_dims(k_pool, v_pool)
    T = int(slot_mapping.numel())
    if k_new.shape != (T, Hkv, D) or v_new.shape != (T, Hkv, D):
        raise ValueError("k_new / v_new must be [T, n_kv_heads, head_dim] matching slot_mapping")
    dt = k_pool.dtype
    opts = make_opts(_block_stride_bytes(k_pool, v_pool))
    st = lib.paged_kv_write_ex(_dev(k_new, "k_new", dt), _dev(v_new, "v_new", dt),
                               _dev(slot_mapping, "slot_mapping", torch.int64), T, _pool(k_pool, "k_pool", dt),
                               _pool(v_pool, "v_pool", dt), NB, S, Hkv, D, _code(dt), ctypes.byref(opts),
                               _stream(stream))
    _check("paged_kv_write", st)


_ws_cache: dict = {}


def decode_workspace_size(batch: int, block_table_stride: int, block_size: int, n_q_heads: int,
                          n_kv_heads: int, head_dim: int, partition_tokens: int = 0) -> int:
    """Split-K workspace bytes for these sizes on the current device (0: never splits)."""
    lib = load_library()
    opts = make_opts(partition_tokens=partition_tokens)
    return int(lib.paged_attention_decode_workspace_size_ex(batch, block_table_stride, block_size, n_q_heads,
                                                            n_kv_heads, head_dim, ctypes.byref(opts)))


def decode_split_plan(batch: int, block_table_stride: int, block_size: int, n_q_heads: int, n_kv_heads: int,
                      head_dim: int, partition_tokens: int = 0, sm_count: int = 152) -> tuple:
    """(partition tokens, partitions per full row, workspace bytes) of the split-K plan on a device
    with ``sm_count`` SMs (host only)."""
    lib = load_library()
    pt, mp, wb = _i32(0), _i32(0), _sz(0)
    _check("pa_decode_split_plan", lib.pa_decode_split_plan(batch, block_table_stride, block_size, n_q_heads,
                                                            n_kv_heads, head_dim, partition_tokens, sm_count,
                                                            ctypes.byref(pt), ctypes.byref(mp), ctypes.byref(wb)))
    return pt.value, mp.value, wb.value


def _workspace(device: torch.device, nbytes: int, stream) -> torch.Tensor | None:
    """The binding's own split-K workspace, one per (device, stream): calls on one stream run in
    order and may share it; calls on different streams may overlap and must not."""
    if nbytes == 0:
        return None
    key = (device.index if device.index is not None else torch.cuda.current_device(), _stream(stream))
    with _lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
            _ws_cache[key] = buf
    return buf


def _decode_args(q, k_pool, v_pool, block_table, context_lens):
    NB, S, Hkv, D = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or q.shape[2] != D:
        raise ValueError("q must be [batch, n_q_heads, head_dim]")
    B, Hq = int(q.shape[0]), int(q.shape[1])
    if block_table.dim() != 2 or block_table.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_table must be [batch, max_blocks] and context_lens [batch]")
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    return NB, S, Hkv, D, B, Hq


def _resolve_workspace(workspace, q, B, bt_stride, S, Hq, Hkv, D, partition_tokens, stream):
    if isinstance(workspace, str) and workspace == "auto":
        ws = _workspace(q.device, decode_workspace_size(B, bt_stride, S, Hq, Hkv, D, partition_tokens), stream)
    else:
        ws = workspace
    return (_dev(ws, "workspace", torch.uint8) if ws is not None else None), (int(ws.numel()) if ws is not None else 0)


def paged_attention_decode(q, k_pool, v_pool, block_table, context_lens, scale=None, out=None,
                           workspace="auto", stream=None, decode_kernel=0, partition_tokens=0):
    """Decode attention: ``q [B, Hq, D]`` over the paged context of each sequence -> ``out [B, Hq, D]``.

    ``workspace``: "auto" (a cached device buffer of the size the library asks for), None (no
    split-K), or a caller-owned uint8 CUDA tensor.  ``decode_kernel`` (0 auto, 1 CUDA cores, 2
    tensor cores) and ``partition_tokens`` (0 automatic) are per-call options."""
    lib = load_library()
    NB, S, Hkv, D, B, Hq = _decode_args(q, k_pool, v_pool, block_table, context_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = k_pool.dtype
    if out is None:
        out = torch.empty_like(q)
    bt_stride = int(block_table.stride(0))
    ws_ptr, ws_bytes = _resolve_workspace(workspace, q, B, bt_stride, S, Hq, Hkv, D, partition_tokens, stream)
    opts = make_opts(_block_stride_bytes(k_pool, v_pool), decode_kernel=decode_kernel,
                     partition_tokens=partition_tokens)
    st = lib.paged_attention_decode_ex(_dev(out, "out", dt), _dev(q, "q", dt), _pool(k_pool, "k_pool", dt),
                                       _pool(v_pool, "v_pool", dt),
                                       _dev(block_table, "block_table", torch.int32, contiguous=False), bt_stride,
                                       _dev(context_lens, "context_lens", torch.int32), B, NB, S, float(scale),
                                       Hq, Hkv, D, _code(dt), ws_ptr, ws_bytes, ctypes.byref(opts), _stream(stream))
    _check("paged_attention_decode", st)
    return out


def paged_attention_decode_fused(q, k_new, v_new, slot_mapping, k_pool, v_pool, block_table, context_lens,
                                 scale=None, out=None, workspace="auto", stream=None, decode_kernel=0,
                                 partition_tokens=0):
    """Write each sequence's new token (row b of ``k_new, v_new [B, Hkv, D]``) to
    ``slot_mapping[b]`` — the slot of its last context position — and attend, in one launch.
    Same result as :func:`paged_kv_write` followed by :func:`paged_attention_decode`."""
    lib = load_library()
    NB, S, Hkv, D, B, Hq = _decode_args(q, k_pool, v_pool, block_table, context_lens)
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or slot_mapping.numel() != B:
        raise ValueError("k_new / v_new must be [batch, n_kv_heads, head_dim] and slot_mapping [batch]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = k_pool.dtype
    if out is None:
        out = torch.empty_like(q)
    bt_stride = int(block_table.stride(0))
    ws_ptr, ws_bytes = _resolve_workspace(workspace, q, B, bt_stride, S, Hq, Hkv, D, partition_tokens, stream)
    opts = make_opts(_block_stride_bytes(k_pool, v_pool), decode_kernel=decode_kernel,
                     partition_tokens=partition_tokens)
    st = lib.paged_attention_decode_fused_ex(
        _dev(out, "out", dt), _dev(q, "q", dt), _dev(k_new, "k_new", dt), _dev(v_new, "v_new", dt),
        _dev(slot_mapping, "slot_mapping", torch.int64), _pool(k_pool, "k_pool", dt), _pool(v_pool, "v_pool", dt),
        _dev(block_table, "block_table", torch.int32, contiguous=False), bt_stride,
        _dev(context_lens, "context_lens", torch.int32), B, NB, S, float(scale), Hq, Hkv, D, _code(dt),
        ws_ptr, ws_bytes, ctypes.byref(opts), _stream(stream))
    _check("paged_attention_decode_fused", st)
    return out


PA_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024


def paged_attention_decode_static_scratch(q, k_pool, v_pool, block_table, context_lens, scale=None, out=None,
                                          stream=None):
    """Decode attention for callers that cannot allocate device memory: same result as
    :func:`paged_attention_decode` (contiguous pools, default options), with the split-K scratch
    taken from the library's own fixed device array (PA_STATIC_SCRATCH_BYTES per device) instead of
    a caller workspace.  Calls that overlap on the GPU share that array and race; serialize them on
    one stream."""
    lib = load_library()
    NB, S, Hkv, D, B, Hq = _decode_args(q, k_pool, v_pool, block_table, context_lens)
    if _block_stride_bytes(k_pool, v_pool) != 0:
        raise ValueError("paged_attention_decode_static_scratch takes contiguous pools")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = k_pool.dtype
    if out is None:
        out = torch.empty_like(q)
    st = lib.paged_attention_decode_static_scratch(
        _dev(out, "out", dt), _dev(q, "q", dt), _pool(k_pool, "k_pool", dt), _pool(v_pool, "v_pool", dt),
        _dev(block_table, "block_table", torch.int32, contiguous=False), int(block_table.stride(0)),
        _dev(context_lens, "context_lens", torch.int32), B, NB, S, float(scale), Hq, Hkv, D, _code(dt),
        _stream(stream))
    _check("paged_attention_decode_static_scratch", st)
    return out


def paged_attention_prefill(q, query_start_loc, k_pool, v_pool, block_table, context_lens, scale=None,
                            out=None, stream=None, prefill_kernel=0):
    """Causal chunked prefill: ``q [total_q, Hq, D]`` (chunks delimited by ``query_start_loc``) over
    each sequence's paged context -> ``out [total_q, Hq, D]``.  ``prefill_kernel``: 0 auto, 1 CUDA
    cores, 2 tcgen05."""
    lib = load_library()
    NB, S, Hkv, D = _pool_dims(k_pool, v_pool)
    if q.dim() != 3 or q.shape[2] != D:
        raise ValueError("q must be [total_q, n_q_heads, head_dim]")
    total_q, Hq = int(q.shape[0]), int(q.shape[1])
    B = int(context_lens.numel())
    if query_start_loc.numel() != B + 1 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("query_start_loc must be [batch + 1] and block_table [batch, max_blocks]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = k_pool.dtype
    if out is None:
        out = torch.empty_like(q)
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    opts = make_opts(_block_stride_bytes(k_pool, v_pool), prefill_kernel=prefill_kernel)
    st = lib.paged_attention_prefill_ex(_dev(out, "out", dt), _dev(q, "q", dt),
                                        _dev(query_start_loc, "query_start_loc", torch.int32), total_q,
                                        _pool(k_pool, "k_pool", dt), _pool(v_pool, "v_pool", dt),
                                        _dev(block_table, "block_table", torch.int32, contiguous=False),
                                        int(block_table.stride(0)), _dev(context_lens, "context_lens", torch.int32),
                                        B, NB, S, float(scale), Hq, Hkv, D, _code(dt), ctypes.byref(opts),
                                        _stream(stream))
    _check("paged_attention_prefill", st)
    return out


def copy_blocks(k_pool, v_pool, block_pairs, stream=None):
    """Copy-on-write block copies: for each ``(src, dst)`` row of int64 ``block_pairs [n, 2]``."""
    lib = load_library()
    NB, S, Hkv, D = _pool_dims(k_pool, v_pool)
    n = int(block_pairs.shape[0]) if block_pairs.numel() else 0
    if block_pairs.numel() and (block_pairs.dim() != 2 or block_pairs.shape[1] != 2):
        raise ValueError("block_pairs must be [n, 2]")
    block_bytes = S * Hkv * D * k_pool.element_size()
    opts = make_opts(_block_stride_bytes(k_pool, v_pool))
    st = lib.copy_blocks_ex(_pool(k_pool, "k_pool"), _pool(v_pool, "v_pool"),
                            _dev(block_pairs, "block_pairs", torch.int64) if n else None, n, NB, block_bytes,
                            ctypes.byref(opts), _stream(stream))
    _check("copy_blocks", st)


def swap_blocks(dst_k_pool, dst_v_pool, src_k_pool, src_v_pool, block_pairs, stream=None):
    """Copy block ``src`` of the source pools to block ``dst`` of the destination pools for every
    ``(src, dst)`` row of int64 ``block_pairs [n, 2]``.  Pools may be CUDA tensors or pinned CPU
    tensors (``pin_memory()``) and share one block stride; ``block_pairs`` a CUDA tensor or a
    pinned CPU tensor."""
    lib = load_library()
    if dst_k_pool.shape[1:] != src_k_pool.shape[1:] or dst_k_pool.dtype != src_k_pool.dtype:
        raise ValueError("source and destination pools must share block shape and dtype")
    for name, t in (("dst_k_pool", dst_k_pool), ("dst_v_pool", dst_v_pool), ("src_k_pool", src_k_pool),
                    ("src_v_pool", src_v_pool)):
        _pool(t, name, host_ok=True)
    stride = _block_stride_bytes(src_k_pool, src_v_pool)
    if _block_stride_bytes(dst_k_pool, dst_v_pool) != stride:
        raise ValueError("source and destination pools must share one block stride")
    if not block_pairs.is_contiguous():
        raise ValueError("block_pairs must be contiguous")
    if not block_pairs.is_cuda and not block_pairs.is_pinned():
        raise ValueError("block_pairs must be a CUDA tensor or pinned host memory")
    n = int(block_pairs.shape[0]) if block_pairs.numel() else 0
    if block_pairs.dtype != torch.int64 or (n and (block_pairs.dim() != 2 or block_pairs.shape[1] != 2)):
        raise ValueError("block_pairs must be int64 [n, 2]")
    block_bytes = int(src_k_pool[0].numel()) * src_k_pool.element_size()
    opts = make_opts(stride)
    st = lib.swap_blocks_ex(dst_k_pool.data_ptr(), dst_v_pool.data_ptr(), int(dst_k_pool.shape[0]),
                            src_k_pool.data_ptr(), src_v_pool.data_ptr(), int(src_k_pool.shape[0]),
                            block_pairs.data_ptr() if n else None, n, block_bytes, ctypes.byref(opts),
                            _stream(stream))
    _check("swap_blocks", st)


def paged_attention_lse_merge(part_max, part_sum, part_acc, out_dtype=torch.bfloat16, out=None, stream=None):
    """Merge split-K partials ``part_max, part_sum [rows, P]`` and ``part_acc [rows, P, D]`` (fp32,
    log2 domain) -> ``out [rows, D]``."""
    lib = load_library()
    rows, P, D = (int(x) for x in part_acc.shape)
    if out is None:
        out = torch.empty((rows, D), dtype=out_dtype, device=part_acc.device)
    st = lib.paged_attention_lse_merge(_dev(out, "out", out.dtype), _dev(part_max, "part_max", torch.float32),
                                       _dev(part_sum, "part_sum", torch.float32),
                                       _dev(part_acc, "part_acc", torch.float32), rows, P, D, _code(out.dtype),
                                       _stream(stream))
    _check("paged_attention_lse_merge", st)
    return out


def set_checked_mode(on: bool):
    """Checked mode (host-side validation of every index array before each launch), process-wide."""
    _check("pa_set_checked_mode", load_library().pa_set_checked_mode(1 if on else 0))


def set_option(option: int, value: int):
    _check("pa_set_option", load_library().pa_set_option(option, int(value)))


def get_option(option: int) -> int:
    return int(load_library().pa_get_option(option))


def device_error_flags(clear: bool = True, stream=None) -> int:
    v = load_library().pa_device_error_flags(1 if clear else 0, _stream(stream))
    if v < 0:
        _check("pa_device_error_flags", v)
    return v


def selftest_bounded_wait(limit_ns: int, stream=None, clear: bool = True) -> tuple:
    """Run the bounded-wait self-test (see pa_selftest_bounded_wait) and return (error flags,
    warp 0's wait in ns, warp 1's wait in ns); the flags are read and, with ``clear``, reset."""
    dev = torch.device("cuda", torch.cuda.current_device())
    elapsed = torch.zeros(2, dtype=torch.int64, device=dev)
    _check("pa_selftest_bounded_wait",
           load_library().pa_selftest_bounded_wait(int(limit_ns), elapsed.data_ptr(), _stream(stream)))
    flags = device_error_flags(clear=clear, stream=stream)
    e = elapsed.cpu()
    return flags, int(e[0]), int(e[1])


def launch_count() -> int:
    return int(load_library().pa_launch_count())


def version() -> str:
    return load_library().pa_version().decode()
