"""The C ABI: the library builds, loads without a GPU and exports every
entry point include/dsa.h declares; host-side argument checks answer
synchronously without touching a device."""
import ctypes
import os
import re

import pytest

from dsa_sparse_attention_index_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"dsa_index_scores", "dsa_topk", "sparse_mla_decode", "dsa_decode_step"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dsa.h but not exported"
    assert names == set(binding.EXPORTS)


def test_version_and_status_strings(lib):
    assert lib.dsa_api_version() == 4
    for code in range(7):
        assert binding.status_string(code).startswith("DSA_")
    assert "unknown" in binding.status_string(99)


def test_host_validation_without_device(lib):
    B = binding
    # null cache / batch descriptors
    assert lib.dsa_index_scores(None, None, None, None, None, 0, None, None) == B.ERR_INVALID_ARG
    c = B.PagedCacheT(None, 45312, 0, 36864, 64, 10, 0, 1.0)
    b = B.BatchT(None, None, 1, 1, 1, 100)
    assert lib.dsa_index_scores(ctypes.byref(c), ctypes.byref(b), None, None, None, 100, None, None) == B.ERR_INVALID_ARG
    c.base = 128 * 1000  # fake, aligned, never dereferenced by the host checks
    c.block_size = 32
    assert lib.dsa_index_scores(ctypes.byref(c), ctypes.byref(b), None, None, None, 100, None, None) == B.ERR_UNSUPPORTED
    c.block_size = 64
    c.row_stride = 45312 + 64  # not a multiple of 128
    assert lib.sparse_mla_decode(ctypes.byref(c), ctypes.byref(b), None, None, 2048, 1.0, None, None, None, 0, None,
                                 None) == B.ERR_INVALID_ARG
    c.row_stride = 45312
    b.block_table, b.seq_lens = 128 * 2000, 128 * 3000  # fake device pointers, never dereferenced here
    for nq in (5, 2049, 0):  # > 4 rows must come in groups of 4; at most 2048; at least 1
        b.queries_per_seq = nq
        assert lib.dsa_decode_step(ctypes.byref(c), ctypes.byref(b), None, None, None, 2048, 1.0, None, None, None,
                                   0, None, None, None, 0, None, None) == B.ERR_UNSUPPORTED
    b.queries_per_seq = 2
    c.key_format = B.KEY_MXFP4  # MXFP4 keys: one row per sequence
    c.row_stride, c.index_off = 41216, 36864
    assert lib.dsa_index_scores(ctypes.byref(c), ctypes.byref(b), None, None, None, 100, None,
                                None) == B.ERR_UNSUPPORTED
    c.key_format, c.row_stride = B.KEY_FP8_E4M3, 45312
    assert lib.dsa_topk(None, 0, None, 1, 10, 0, None, None, 0, None, None) == B.ERR_INVALID_ARG  # k = 0
    assert lib.dsa_topk(None, 0, None, 1, 10, 4096, None, None, 0, None, None) == B.ERR_INVALID_ARG  # k > 2048
    st = 128 * 4000  # fake device status pointer
    # DCP merge: at most 8 shards, at most 65,536 tokens per shard and row
    assert lib.dsa_dcp_topk(None, 0, None, 1, 10, 2048, 9, None, None, None, 0, st, None) == B.ERR_UNSUPPORTED
    assert lib.dsa_dcp_topk(None, 0, None, 1, 2 * 65536 + 1, 2048, 2, None, None, None, 0, st,
                            None) == B.ERR_UNSUPPORTED
    assert lib.dsa_dcp_topk(None, 0, None, 1, 10, 2048, 0, None, None, None, 0, st, None) == B.ERR_INVALID_ARG
    assert lib.dsa_dcp_topk(128, 16, 256, 1, 10, 2048, 8, 512, None, None, 0, st, None) == B.ERR_WORKSPACE
    # latent formats: FP8 (0) and NVFP4 (1, 352-byte records: a smaller row fits); nothing else
    c.latent_format = 2
    assert lib.dsa_index_scores(ctypes.byref(c), ctypes.byref(b), 1024, 2048, 4096, 104, st,
                                None) == B.ERR_INVALID_ARG
    c.latent_format, c.row_stride = B.LATENT_NVFP4, 64 * 352 + 64 * 132 + 128
    c.index_off = 64 * 352 + 64                     # not a multiple of 128
    assert lib.dsa_index_scores(ctypes.byref(c), ctypes.byref(b), 1024, 2048, 4096, 104, st,
                                None) == B.ERR_INVALID_ARG
    c.latent_format, c.row_stride, c.index_off = 0, 45312, 36864
    # rows longer than a cluster holds need the two-level workspace: NULL, too small or
    # misaligned is refused before anything is launched
    need = lib.dsa_topk_workspace_size(4, 1 << 20, 2048)
    assert lib.dsa_topk(128, 1 << 20, 256, 4, 1 << 20, 2048, 512, None, 0, st, None) == B.ERR_WORKSPACE
    assert lib.dsa_topk(128, 1 << 20, 256, 4, 1 << 20, 2048, 512, 1 << 20, need - 1, st, None) == B.ERR_WORKSPACE
    assert lib.dsa_topk(128, 1 << 20, 256, 4, 1 << 20, 2048, 512, (1 << 20) + 16, need, st, None) == B.ERR_WORKSPACE
    assert lib.dsa_topk(128, (1 << 20) + 2, 256, 4, 1 << 20, 2048, 512, 1 << 20, need, st, None) == B.ERR_INVALID_ARG
    # the no-allocation entry point: at most 64 rows
    assert lib.dsa_topk_noalloc(128, 1 << 20, 256, 65, 1 << 20, 2048, 512, st, None) == B.ERR_UNSUPPORTED
    # bf16 scores: rows of a multiple of 8 elements
    assert lib.dsa_topk_bf16(128, 12, 256, 1, 10, 2048, 512, st, None) == B.ERR_INVALID_ARG
    assert lib.dsa_topk_bf16(128, 16, 256, 1, 10, 0, 512, st, None) == B.ERR_INVALID_ARG
    assert lib.dsa_index_scores_bf16(ctypes.byref(c), ctypes.byref(b), 1024, 2048, 4096, 100, st,
                                     None) == B.ERR_INVALID_ARG
    # DCP LSE combine: 1..8 shards, aligned pointers, a workspace of the stated size
    b.queries_per_seq = 1
    dm = lambda shards, q, out, ws, n: lib.dsa_dcp_sparse_mla(ctypes.byref(c), ctypes.byref(b), q, 256, 2048, shards,
                                                              1.0, out, 512, None, None, ws, n, st, None)
    assert dm(9, 1024, 2048, None, 0) == B.ERR_UNSUPPORTED
    assert dm(0, 1024, 2048, None, 0) == B.ERR_INVALID_ARG
    assert dm(8, 1032, 2048, None, 0) == B.ERR_INVALID_ARG        # q_mla not 16-byte aligned
    assert dm(8, 1024, 2052, None, 0) == B.ERR_INVALID_ARG        # out not 8-byte aligned
    assert dm(8, 1024, 2048, 4096, 100) == B.ERR_WORKSPACE
    # partial outputs, when given, 8-byte aligned like the output
    assert lib.dsa_dcp_sparse_mla(ctypes.byref(c), ctypes.byref(b), 1024, 256, 2048, 4, 1.0, 2048, 512, 3076, None,
                                  4096, 1 << 40, st, None) == B.ERR_INVALID_ARG
    # bf16 fused step: a caller's score buffer needs a row stride that is a multiple of 8
    assert lib.dsa_decode_step_bf16(ctypes.byref(c), ctypes.byref(b), 1024, 2048, 4096, 2048, 1.0, 8192, 512, 16384,
                                    100, None, None, 4096, 1 << 40, st, None) == B.ERR_INVALID_ARG


def test_workspace_sizes(lib):
    b = binding.BatchT(None, None, 2560, 32, 1, 163840)
    ws = lib.dsa_workspace_size(ctypes.byref(b), 2048)
    assert ws >= 32 * 163840 * 4  # holds the scores
    assert lib.dsa_topk_workspace_size(4, 1 << 20, 2048) > 0
    # two levels for long rows: at least 7 segments' candidates, their scores and tokens
    assert lib.dsa_topk_workspace_size(4, 1 << 20, 2048) >= 2 * 4 * 7 * 2048 * 4
    assert lib.sparse_mla_workspace_size(32, 2048) >= 32 * 96 * 512 * 2  # fp16 partials
    assert lib.dsa_topk_workspace_size(32, 163840, 2048) == 0  # rows held in shared memory
    assert lib.dsa_topk_workspace_size(4, 100, 0) == 0
    # DCP: one candidate slot of max(ceil(1.5 k / W), k) words per (row, shard), plus counters
    assert lib.dsa_dcp_topk_workspace_size(32, 2048, 8) >= 32 * 8 * 2048 * 4
    assert lib.dsa_dcp_topk_workspace_size(4, 2048, 1) >= 4 * 3072 * 4
    assert lib.dsa_dcp_topk_workspace_size(4, 2048, 9) == 0
    # DCP LSE combine: the grouped indices plus fp16 partials of 2 pieces per shard (k = 2048)
    assert lib.dsa_dcp_sparse_mla_workspace_size(32, 2048, 8) >= 32 * 16 * 96 * 512 * 2 + 32 * 2048 * 4
    assert lib.dsa_dcp_sparse_mla_workspace_size(4, 1024, 3) >= 4 * 3 * 96 * 512 * 2
    assert lib.dsa_dcp_sparse_mla_workspace_size(4, 2048, 9) == 0
    # batch-invariant mode: 512-token chunks, so the partials of 200 rows need 4 slots a row
    assert lib.dsa_batch_invariant(1) == 0
    try:
        assert lib.sparse_mla_workspace_size(200, 2048) >= 200 * 4 * 96 * 512 * 2
    finally:
        assert lib.dsa_batch_invariant(0) == 1
    assert lib.sparse_mla_workspace_size(200, 2048) < 200 * 4 * 96 * 512 * 4


def test_oracle_and_product_share_no_code():
    """The product (package and CUDA sources) never imports or includes the
    oracle, and the oracle never imports the product."""
    pkg = os.path.join(ROOT, "dsa_sparse_attention_index_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), f
                assert not re.search(r'#include\s+[<"][^>"]*oracle', src), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+dsa_sparse_attention_index_gb300\b", src, flags=re.M), f
            assert not re.search(r'#include\s+[<"][^>"]*(csrc|dsa\.h|common\.cuh)', src), f


def test_frontend_host_validation_without_device(lib):
    """The fused front end refuses a compressed-query width that is not a
    multiple of 64 (DSA_ERR_UNSUPPORTED) and missing or misaligned buffers
    (DSA_ERR_INVALID_ARG) before any launch; the step variant checks its
    workspace the same way."""
    B = binding
    c = B.PagedCacheT(128 * 1000, 45312, 0, 36864, 64, 10, 0, 1.0)
    b = B.BatchT(128 * 2000, 128 * 3000, 4, 1, 1, 100)
    st = 128 * 4000
    fake = 128 * 5000
    args = lambda rank, cq=fake, g=fake, eps=1e-6: (ctypes.byref(c), ctypes.byref(b), cq, rank, g, eps, fake, fake,
                                                     fake, fake, fake, fake, None, st, None)
    assert lib.dsa_index_frontend(*args(1000)) == B.ERR_UNSUPPORTED
    assert lib.dsa_index_frontend(*args(0)) == B.ERR_UNSUPPORTED
    assert lib.dsa_index_frontend(*args(1536, cq=None)) == B.ERR_INVALID_ARG
    assert lib.dsa_index_frontend(*args(1536, g=fake + 2)) == B.ERR_INVALID_ARG   # gamma not 16-B aligned
    assert lib.dsa_index_frontend(*args(1536, eps=-1.0)) == B.ERR_INVALID_ARG
    need = lib.dsa_frontend_workspace_size(ctypes.byref(b), 2048)
    assert need >= lib.dsa_workspace_size(ctypes.byref(b), 2048) + 4096
    assert lib.dsa_decode_step_frontend(ctypes.byref(c), ctypes.byref(b), fake, 1536, fake, 1e-6, fake, fake, fake,
                                        fake, fake, 2048, 1.0, fake, fake, None, 0, None, None, fake, need - 1, st,
                                        None) == B.ERR_WORKSPACE
