"""Host-only checks of the C ABI: the library builds/loads, exports every function include/*.h
declares, and rejects bad arguments before touching a GPU.  No compute call is made here."""
import ctypes
import glob
import os
import re

import pytest

import pagedattention_kv_cache_paged_gb300 as pa
from pagedattention_kv_cache_paged_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^PA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_abi.LIB_PATH):
        from pagedattention_kv_cache_paged_gb300 import build
        build.build()
    return pa.load_library()


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
        assert n in _abi.SIGNATURES, n
    assert set(_abi.SIGNATURES) == set(names)


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.pa_version()
    assert lib.pa_status_string(pa.PA_ERANGE) != lib.pa_status_string(0)


def test_options_validate(lib):
    assert lib.pa_set_option(999, 1) == pa.PA_EINVAL
    assert lib.pa_set_option(pa.PA_OPT_CHECKED, 2) == pa.PA_EINVAL
    assert lib.pa_set_option(pa.PA_OPT_DECODE_KERNEL, 3) == pa.PA_EINVAL
    assert lib.pa_set_option(pa.PA_OPT_PARTITION_TOKENS, 256) == 0
    assert lib.pa_get_option(pa.PA_OPT_PARTITION_TOKENS) == 256
    assert lib.pa_set_option(pa.PA_OPT_PARTITION_TOKENS, 0) == 0
    assert lib.pa_set_option(pa.PA_OPT_CLUSTER_MERGE, 2) == pa.PA_EINVAL
    assert lib.pa_get_option(pa.PA_OPT_CLUSTER_MERGE) == 0
    assert lib.pa_set_option(pa.PA_OPT_KV_LAYOUT, 2) == pa.PA_EINVAL
    assert lib.pa_get_option(pa.PA_OPT_KV_LAYOUT) == pa.KV_LAYOUT_SEPARATE


def test_unified_layout_requires_v_to_be_the_v_half_of_block_0(lib):
    """With unified K/V blocks the V view must start one K half after the K view; any other pair
    of pointers is refused before anything is launched (the pointers are never dereferenced)."""
    half = 16 * 2 * 64 * 2
    k = 1 << 20
    assert lib.pa_set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED) == 0
    try:
        assert lib.copy_blocks(k, k + 2 * half, 1 << 24, 1, 4, half, None) == pa.PA_EINVAL
        assert lib.copy_blocks(k + half, k, 1 << 24, 1, 4, half, None) == pa.PA_EINVAL
        assert lib.paged_kv_write(1 << 24, 1 << 24, 1 << 24, 1, k, k + 16, 4, 16, 2, 64, pa.PA_BF16, None) \
            == pa.PA_EINVAL
        args = [1 << 24, 1 << 24, k, k + half // 2, 1 << 24, 4, 1 << 24, 2, 8, 16, 1.0]
        assert lib.paged_attention_decode(*args, 8, 2, 64, pa.PA_BF16, None, 0, None) == pa.PA_EINVAL
        assert lib.swap_blocks(k, k + half, 4, k, k + 3 * half, 4, 1 << 24, 1, half, None) == pa.PA_EINVAL
    finally:
        assert lib.pa_set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_SEPARATE) == 0


def test_argument_errors_are_returned_before_any_launch(lib):
    n = None
    # bad dtype
    assert lib.paged_kv_write(n, n, n, 1, n, n, 4, 16, 2, 64, 7, n) == pa.PA_EDTYPE
    # zero tokens is a no-op
    assert lib.paged_kv_write(n, n, n, 0, n, n, 4, 16, 2, 64, pa.PA_BF16, n) == 0
    # null pointers
    assert lib.paged_kv_write(n, n, n, 3, n, n, 4, 16, 2, 64, pa.PA_BF16, n) == pa.PA_EINVAL
    # heads not divisible / unsupported group / unsupported head_dim / bad block size
    args = [n, n, n, n, n, 4, n, 2, 8, 16, 1.0]
    assert lib.paged_attention_decode(*args, 6, 4, 64, pa.PA_BF16, n, 0, n) == pa.PA_EINVAL
    assert lib.paged_attention_decode(*args, 96, 3, 64, pa.PA_BF16, n, 0, n) == pa.PA_EUNSUPPORTED  # group 32
    assert lib.paged_attention_decode(*args, 36, 3, 64, pa.PA_BF16, n, 0, n) == pa.PA_EUNSUPPORTED  # group 12
    assert lib.paged_attention_decode(*args, 8, 2, 96, pa.PA_BF16, n, 0, n) == pa.PA_EUNSUPPORTED
    bad_bs = [n, n, n, n, n, 4, n, 2, 8, 12, 1.0]
    assert lib.paged_attention_decode(*bad_bs, 8, 2, 64, pa.PA_BF16, n, 0, n) == pa.PA_EUNSUPPORTED
    # batch 0 is a no-op
    zero = [n, n, n, n, n, 4, n, 0, 8, 16, 1.0]
    assert lib.paged_attention_decode(*zero, 8, 2, 64, pa.PA_BF16, n, 0, n) == 0
    # copy_blocks: block bytes must be a multiple of 16
    assert lib.copy_blocks(n, n, n, 1, 4, 24, n) == pa.PA_EINVAL
    assert lib.copy_blocks(n, n, n, 0, 4, 32, n) == 0
    # merge
    assert lib.paged_attention_lse_merge(n, n, n, n, 4, 0, 64, pa.PA_BF16, n) == pa.PA_EINVAL
    assert lib.paged_attention_lse_merge(n, n, n, n, 4, 2, 80, pa.PA_BF16, n) == pa.PA_EUNSUPPORTED


def test_workspace_size_follows_the_partition_plan(lib):
    f = lib.paged_attention_decode_workspace_size
    # short tables never split
    assert f(64, 8, 16, 32, 8, 128) == 0
    # 4096-token tables at the default 1024-token partitions: 4 partitions of (128 + 2) floats
    ws = f(64, 256, 16, 32, 8, 128)
    assert ws >= 64 * 32 * 4 * 130 * 4
    assert ws % 16 == 0
    assert lib.pa_set_option(pa.PA_OPT_PARTITION_TOKENS, 2048) == 0
    assert f(64, 256, 16, 32, 8, 128) < ws
    assert lib.pa_set_option(pa.PA_OPT_PARTITION_TOKENS, 0) == 0


def _expected_workspace(batch, stride, bs, hq, hkv, d, part=0):
    """The documented split-K plan: automatic partitions give about one wave of 456 decode CTAs when
    every row is as long as its table allows, clamped to [256, 1024] tokens and rounded up to the
    block size; slots = partitions + 1; acc, max, sum and per-sequence slot counts, 16-byte aligned."""
    max_len = stride * bs
    if part <= 0:
        part = min(max(-(-batch * hkv * max_len // 456), 256), 1024)
    part = -(-part // bs) * bs
    if part >= max_len:
        return 0
    slots = -(-max_len // part) + 1
    n = batch * hq * slots
    up16 = lambda x: (x + 15) // 16 * 16
    return n * d * 4 + 2 * up16(n * 4) + up16(batch * 4)


@pytest.mark.parametrize("shape", [(64, 256, 16, 32, 8, 128), (1, 128, 16, 12, 12, 64), (8, 128, 16, 12, 12, 64),
                                   (4, 8192, 16, 32, 8, 128), (64, 8, 16, 32, 8, 128), (3, 40, 32, 16, 1, 64)])
def test_automatic_split_plan(lib, shape):
    f = lib.paged_attention_decode_workspace_size
    assert f(*shape) == _expected_workspace(*shape)
    assert lib.pa_set_option(pa.PA_OPT_PARTITION_TOKENS, 512) == 0
    try:
        assert f(*shape) == _expected_workspace(*shape, part=512)
    finally:
        assert lib.pa_set_option(pa.PA_OPT_PARTITION_TOKENS, 0) == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    kp = torch.zeros((4, 16, 2, 64))
    with pytest.raises(ValueError):
        pa.paged_kv_write(torch.zeros((1, 2, 64)), torch.zeros((1, 2, 64)), torch.zeros(1, dtype=torch.int64),
                          kp, kp.clone())


def test_library_source_has_no_oracle_dependency():
    pkg = os.path.join(ROOT, "pagedattention_kv_cache_paged_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path).read()
            assert "oracle" not in text.replace("no oracle", ""), path
