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


def test_the_only_process_wide_option_is_checked_mode(lib):
    assert lib.pa_set_option(999, 1) == pa.PA_EINVAL
    for legacy in range(2, 8):  # tuning and layout choices are per-call options now
        assert lib.pa_set_option(legacy, 0) == pa.PA_EINVAL
        assert lib.pa_get_option(legacy) == pa.PA_EINVAL
    assert lib.pa_set_option(pa.PA_OPT_CHECKED, 2) == pa.PA_EINVAL
    assert lib.pa_set_checked_mode(2) == pa.PA_EINVAL
    assert lib.pa_set_checked_mode(1) == 0
    assert lib.pa_get_option(pa.PA_OPT_CHECKED) == 1
    assert lib.pa_set_checked_mode(0) == 0
    assert lib.pa_get_option(pa.PA_OPT_CHECKED) == 0


def _opts(**kw):
    return ctypes.byref(pa.make_opts(**kw))


def test_per_call_options_are_validated_before_any_launch(lib):
    """Bad per-call options are refused before anything touches a device (the pointers are never
    dereferenced)."""
    block = 16 * 2 * 64 * 2
    k = 1 << 20
    bad = [dict(kv_block_stride_bytes=block + 8),  # not a multiple of 16
           dict(kv_block_stride_bytes=block - 16),  # shorter than a block
           dict(kv_block_stride_bytes=-32), dict(decode_kernel=3), dict(prefill_kernel=3),
           dict(partition_tokens=-1), dict(partition_tokens=(1 << 30) + 1)]
    dec = [1 << 24, 1 << 24, k, k + block, 1 << 24, 4, 1 << 24, 2, 8, 16, 1.0, 8, 2, 64, pa.PA_BF16, None, 0]
    for kw in bad:
        o = _opts(**kw)
        assert lib.paged_attention_decode_ex(*dec, o, None) == pa.PA_EINVAL, kw
        assert lib.paged_attention_decode_fused_ex(1 << 24, 1 << 24, 1 << 24, 1 << 24, 1 << 24, k, k + block, 1 << 24,
                                                   4, 1 << 24, 2, 8, 16, 1.0, 8, 2, 64, pa.PA_BF16, None, 0, o,
                                                   None) == pa.PA_EINVAL, kw
        assert lib.paged_attention_prefill_ex(1 << 24, 1 << 24, 1 << 24, 4, k, k + block, 1 << 24, 4, 1 << 24, 2, 8,
                                              16, 1.0, 8, 2, 64, pa.PA_BF16, o, None) == pa.PA_EINVAL, kw
        assert lib.paged_attention_decode_workspace_size_ex(64, 256, 16, 32, 8, 128, o) == 0, kw
    for kw in bad[:3]:
        o = _opts(**kw)
        assert lib.paged_kv_write_ex(1 << 24, 1 << 24, 1 << 24, 1, k, k + block, 4, 16, 2, 64, pa.PA_BF16, o,
                                     None) == pa.PA_EINVAL, kw
        assert lib.copy_blocks_ex(k, k + block, 1 << 24, 1, 4, block, o, None) == pa.PA_EINVAL, kw
        assert lib.swap_blocks_ex(k, k + block, 4, k, k + block, 4, 1 << 24, 1, block, o, None) == pa.PA_EINVAL, kw
    reserved = pa.PaOpts(0, 0, 0, 0, 1)
    assert lib.paged_attention_decode_ex(*dec, ctypes.byref(reserved), None) == pa.PA_EINVAL
    # a null options pointer is the defaults: batch 0 is a no-op
    zero = [None, None, None, None, None, 4, None, 0, 8, 16, 1.0, 8, 2, 64, pa.PA_BF16, None, 0]
    assert lib.paged_attention_decode_ex(*zero, None, None) == 0


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


def test_split_plan_follows_the_partition_rule(lib):
    plan = pa.decode_split_plan
    # short tables never split
    assert plan(64, 8, 16, 32, 8, 128) == (128, 1, 0)
    # 4096-token tables at 1024-token partitions: 4 partitions of (128 + 2) floats per (sequence, head)
    pt, mp, ws = plan(64, 256, 16, 32, 8, 128)
    assert (pt, mp) == (1024, 4)
    assert ws >= 64 * 32 * 4 * 130 * 4 and ws % 16 == 0
    assert plan(64, 256, 16, 32, 8, 128, partition_tokens=2048)[2] < ws
    # invalid sizes
    pt, mp, wb = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_size_t(0)
    args = (ctypes.byref(pt), ctypes.byref(mp), ctypes.byref(wb))
    assert lib.pa_decode_split_plan(0, 256, 16, 32, 8, 128, 0, 152, *args) == pa.PA_EINVAL
    assert lib.pa_decode_split_plan(64, 256, 16, 32, 8, 128, 0, 0, *args) == pa.PA_EINVAL
    assert lib.pa_decode_split_plan(64, 256, 16, 30, 8, 128, 0, 152, *args) == pa.PA_EINVAL
    assert lib.pa_decode_split_plan(64, 256, 16, 32, 8, 128, -4, 152, *args) == pa.PA_EINVAL


def _expected_plan(batch, stride, bs, hq, hkv, d, part=0, sms=152):
    """The documented split-K plan: automatic partitions give at most one wave of decode CTAs (SM
    count x 3, x 2 for groups of 16 query heads) when every row is as long as its table allows —
    floor(wave / rows) partitions per row, at least one — clamped to [256, 1024] tokens and rounded
    up to the block size; the workspace holds acc, max and sum per (sequence, query head,
    partition), each section 16-byte aligned."""
    max_len = stride * bs
    if part <= 0:
        target = sms * (2 if hq // hkv > 8 else 3)
        per_row = max(1, target // (batch * hkv))
        part = min(max(-(-max_len // per_row), 256), 1024)
    part = -(-part // bs) * bs
    if part >= max_len:
        return max_len, 1, 0
    parts = -(-max_len // part)
    n = batch * hq * parts
    up16 = lambda x: (x + 15) // 16 * 16
    return part, parts, n * d * 4 + 2 * up16(n * 4)


@pytest.mark.parametrize("shape", [(64, 256, 16, 32, 8, 128), (1, 128, 16, 12, 12, 64), (8, 128, 16, 12, 12, 64),
                                   (4, 8192, 16, 32, 8, 128), (64, 8, 16, 32, 8, 128), (3, 40, 32, 16, 1, 64),
                                   (2, 512, 16, 64, 4, 128), (1, 64, 16, 16, 1, 128)])
@pytest.mark.parametrize("sms", [152, 148, 132, 20])
def test_automatic_split_plan(lib, shape, sms):
    assert pa.decode_split_plan(*shape, sm_count=sms) == _expected_plan(*shape, sms=sms)
    assert pa.decode_split_plan(*shape, partition_tokens=512, sm_count=sms) == _expected_plan(*shape, part=512,
                                                                                              sms=sms)


def test_groups_of_sixteen_plan_for_two_ctas_per_sm(lib):
    # 4 sequences x 4 KV heads = 16 rows of 16384 tokens: 3 x 152 = 456 CTAs (groups of 8) give 28
    # partitions per row, 586 -> 592 tokens; 2 x 152 = 304 CTAs (groups of 16) give 19, 863 -> 864
    assert pa.decode_split_plan(4, 1024, 16, 32, 4, 128)[:2] == (592, 28)
    assert pa.decode_split_plan(4, 1024, 16, 64, 4, 128)[:2] == (864, 19)


@pytest.mark.parametrize("shape", [(8, 128, 16, 12, 12, 64), (4, 1024, 16, 32, 4, 128), (3, 333, 16, 32, 8, 128),
                                   (5, 999, 16, 40, 8, 128), (1, 8192, 16, 32, 8, 128)])
def test_automatic_plan_never_spills_into_a_second_wave(lib, shape):
    # a grid of rows x partitions that exceeded one wave by a few CTAs would run a second, nearly
    # empty wave as long as the first (batch 8 x 2048 tokens at 12 heads: 5 partitions of 432 tokens
    # made 480 CTAs for 456 slots; 4 of 512 make 384)
    batch, hkv = shape[0], shape[4]
    part, parts, _ = pa.decode_split_plan(*shape, sm_count=152)
    if part > 256 and part < 1024:
        assert batch * hkv * parts <= 152 * 3


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
