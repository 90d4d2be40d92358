"""The C ABI library builds, loads without a GPU, exports every entry point
include/pagedkv.h declares, and rejects bad arguments on the host with a
status code before launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_98_gb300 as pkv
from paged_kv_cache_98_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pkv_reshape_and_cache", "pkv_paged_attention_decode",
                 "pkv_paged_attention_prefill_chunk", "pkv_decode_workspace_size",
                 "pkv_prefill_workspace_size", "pkv_check_errors", "pkv_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pkv_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_status_strings(lib):
    assert pkv.status_string(0) == "ok"
    assert "unsupported" in pkv.status_string(-2)
    assert pkv.version() >= 100


def test_workspace_sizes(lib):
    # one partition: no workspace
    assert pkv.decode_workspace_size(64, 32, 128, 512) == 0
    # 64 x 32 heads x 8 partitions: lse + partial outputs
    heads = 64 * 32 * 8
    want = (-(-heads * 4 // 256) * 256) + (-(-heads * 128 * 4 // 256) * 256)
    assert pkv.decode_workspace_size(64, 32, 128, 4096) == want
    assert pkv.decode_workspace_size(64, 32, 128, 4096, 256) > want


def _decode(lib, **over):
    a = dict(out=256, q=256, k_cache=512, v_cache=512, block_tables=1024, context_lens=2048,
             num_seqs=2, num_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
             max_blocks_per_seq=4, num_blocks=8, max_context_len=64, scale=0.1, q_dtype=1,
             kv_dtype=1, k_scale=1.0, v_scale=1.0, partition_size=0, workspace=None,
             workspace_bytes=0, device_errors=None, stream=None)
    a.update(over)
    return lib.pkv_paged_attention_decode(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=96), -2),
    (dict(block_size=32), -2),
    (dict(num_heads=6, num_kv_heads=4), -1),
    (dict(num_heads=34, num_kv_heads=2), -2),
    (dict(q_dtype=2), -2),
    (dict(q_dtype=0, kv_dtype=1), -2),
    (dict(kv_dtype=2, k_scale=0.0), -1),
    (dict(q=None), -1),
    (dict(out=258), -1),
    (dict(partition_size=24), -1),
    (dict(partition_size=1024), -1),
    (dict(max_context_len=4096), -3),
    (dict(num_seqs=0), 0),
])
def test_decode_argument_validation(lib, over, status):
    assert _decode(lib, **over) == status


def test_reshape_argument_validation(lib):
    f = lib.pkv_reshape_and_cache
    base = [256, 256, 512, 512, 1024, 4, 2, 128, 16, 8, 1, 1, 1.0, 1.0, None, None]
    assert f(*base[:5], 0, *base[6:]) == 0  # nothing to write
    bad = list(base)
    bad[7] = 80
    assert f(*bad) == -2
    bad = list(base)
    bad[0] = None
    assert f(*bad) == -1
    bad = list(base)
    bad[11] = 2
    bad[12] = -1.0
    assert f(*bad) == -1


def test_prefill_argument_validation(lib):
    f = lib.pkv_paged_attention_prefill_chunk
    args = [256, 256, 512, 512, 1024, 2048, None, 1, 10, 10, 8, 2, 128, 16, 4, 8, 64, 0.1, 1, 1,
            1.0, 1.0, None, 0, None, None]
    assert f(*args) == -1  # query_start_loc missing


def _cascade(lib, **over):
    a = dict(out=256, q=256, k_cache=512, v_cache=512, block_tables=1024, context_lens=2048,
             group_start=4096, prefix_lens=8192, num_seqs=2, num_groups=1, num_heads=8,
             num_kv_heads=2, head_dim=128, block_size=16, max_blocks_per_seq=4, num_blocks=8,
             max_context_len=64, max_prefix_len=32, scale=0.1, q_dtype=1, kv_dtype=1,
             k_scale=1.0, v_scale=1.0, workspace=None, workspace_bytes=0, device_errors=None,
             stream=None)
    a.update(over)
    return lib.pkv_paged_attention_decode_cascade(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(group_start=None), -1),
    (dict(prefix_lens=None), -1),
    (dict(max_prefix_len=128), -1),   # longer than max_context_len
    (dict(num_groups=-1), -1),
    (dict(head_dim=96), -2),
    (dict(head_dim=64), -2),          # the cascade runs on the 128-dim tensor-core kernels
    (dict(kv_dtype=2), -2),           # 16-bit caches only
    (dict(q=None), -1),
    (dict(num_seqs=0), 0),
])
def test_cascade_argument_validation(lib, over, status):
    assert _cascade(lib, **over) == status


def test_cascade_workspace_size(lib):
    # two partials per 2048-key chunk of the prefix, then 512-token partitions
    slots = 2 * 3 + 8
    heads = 64 * 32 * slots
    want = (-(-heads * 4 // 256) * 256) + (-(-heads * 128 * 4 // 256) * 256)
    assert pkv.cascade_workspace_size(64, 32, 128, 4096, 5000) == want
    # always a workspace, even for one partition and no prefix
    assert pkv.cascade_workspace_size(1, 8, 128, 16, 0) > 0


def test_tree_argument_validation(lib):
    f = lib.pkv_paged_attention_prefill_tree
    args = [256, 256, 512, 512, 1024, 2048, 4096, 8192, 1, 10, 10, 8, 2, 128, 16, 4, 8, 64, 0.1,
            1, 1, 1.0, 1.0, None, None]
    assert f(*args[:7], None, *args[8:]) == -1  # no mask
    long = list(args)
    long[10] = 65  # max_q_len above 64
    assert f(*long) == -1
    assert f(*args[:8], 0, *args[9:]) == 0  # no sequences


def test_mixed_argument_validation(lib):
    f = lib.pkv_paged_attention_mixed
    # out q k v tables lens qsl | decode seqs total_q max_q H Hkv D bs MB NB max_ctx | scale
    # dtypes scales | prefill_ctas workspace bytes errors stream
    args = [256, 256, 512, 512, 1024, 2048, 4096, 2, 4, 40, 16, 8, 2, 128, 16, 4, 8, 64, 0.1,
            1, 1, 1.0, 1.0, 0, None, 0, None, None]

    def call(**over):
        a = list(args)
        for i, v in over.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a6=None) == -1       # no query_start_loc
    assert call(a7=5) == -1          # more decode rows than sequences
    assert call(a9=1) == -1          # fewer query rows than decode rows
    assert call(a23=-1) == -1        # negative CTA share
    assert call(a7=0, a8=0, a9=0) == 0  # empty batch: nothing launched


def test_mixed_workspace_size(lib):
    # the larger of the decode rows' and the chunks' needs
    d = pkv.decode_workspace_size(32, 32, 128, 8192)
    p = pkv.prefill_workspace_size(2048, 32, 128, 8192, 512)
    assert pkv.mixed_workspace_size(32, 2080, 32, 128, 8192) == max(d, p)


def test_mixed_workspace_is_checked(lib):
    # decode rows over 4096 tokens need split-K workspace: missing or short -> PKV_ERR_WORKSPACE
    f = lib.pkv_paged_attention_mixed
    args = [256, 256, 512, 512, 1024, 2048, 4096, 2, 4, 40, 16, 8, 2, 128, 16, 256, 4096, 4096,
            0.1, 1, 1, 1.0, 1.0, 0, None, 0, None, None]
    assert f(*args) == -3
    short = list(args)
    short[24], short[25] = 256, 512
    assert f(*short) == -3


def test_copy_blocks_argument_checks(lib):
    f = lib.pkv_copy_blocks
    # caches, pairs, num_pairs, Hkv, D, block_size, num_blocks, dtype, errors, stream
    assert f(256, 256, 512, 0, 8, 128, 16, 64, 1, None, None) == 0      # nothing to copy
    assert f(None, 256, 512, 4, 8, 128, 16, 64, 1, None, None) == -1    # no cache
    assert f(264, 256, 512, 4, 8, 128, 16, 64, 1, None, None) == -1    # misaligned cache
    assert f(256, 256, 512, 4, 8, 128, 32, 64, 1, None, None) == -2    # block size 32
    assert f(256, 256, 512, -1, 8, 128, 16, 64, 1, None, None) == -1   # negative count
