"""ctypes binding of libdsa.so — argument marshalling only.

Every entry point here forwards torch CUDA tensors (as raw device pointers)
and the current CUDA stream to the C ABI declared in ``include/dsa.h``; all
arithmetic happens in the library's kernels.  There is no CPU fallback: if
the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_BOUNDS, ERR_TIMEOUT, ERR_CUDA, ERR_WORKSPACE = range(7)
KEY_FP8_E4M3, KEY_MXFP4, KEY_MXFP4_NATIVE = 0, 1, 2
LATENT_FP8_E4M3, LATENT_NVFP4 = 0, 1
BLOCK, IDX_HEADS, IDX_DIM, MLA_HEADS, LATENT, VALUE, MAX_TOPK = 64, 32, 128, 96, 576, 512, 2048


class DsaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        extra = ""
        if code == ERR_CUDA:
            extra = f" [{lib().dsa_last_cuda_error().decode()}]"
        super().__init__(f"{what}: {status_string(code)}{extra}")


class PagedCacheT(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("row_stride", ctypes.c_int64), ("latent_off", ctypes.c_int64),
                ("index_off", ctypes.c_int64), ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("key_format", ctypes.c_int32), ("latent_scale", ctypes.c_float), ("latent_format", ctypes.c_int32)]


class BatchT(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("queries_per_seq", ctypes.c_int32), ("max_seq_len", ctypes.c_int32)]


_lib = None

EXPORTS = ["dsa_api_version", "dsa_status_string", "dsa_last_cuda_error", "dsa_kernel_launches",
           "dsa_translate_pages", "dsa_index_scores", "dsa_index_scores_bf16", "dsa_topk_bf16",
           "dsa_decode_step_bf16",
           "dsa_topk_workspace_size", "dsa_topk", "dsa_topk_noalloc", "dsa_topk_force_multipass", "dsa_topk_paged",
           "dsa_dcp_topk_workspace_size", "dsa_dcp_topk", "sparse_mla_workspace_size",
           "sparse_mla_decode", "dsa_dcp_sparse_mla_workspace_size", "dsa_dcp_sparse_mla", "dsa_batch_invariant",
           "dsa_workspace_size", "dsa_decode_step", "dsa_cache_append", "dsa_quantize_index_query",
           "dsa_index_frontend", "dsa_frontend_workspace_size", "dsa_decode_step_frontend",
           "dsa_selftest_wait_timeout"]


def lib():
    """Load libdsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdsa.so not found at {LIB_PATH}: build it with "
                               "dsa_sparse_attention_index_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        pc, pb = ctypes.POINTER(PagedCacheT), ctypes.POINTER(BatchT)
        sig = {
            "dsa_api_version": (i32, []),
            "dsa_status_string": (ctypes.c_char_p, [i32]),
            "dsa_last_cuda_error": (ctypes.c_char_p, []),
            "dsa_kernel_launches": (ctypes.c_uint64, []),
            "dsa_translate_pages": (i32, [pc, pb, P, P, P, P]),
            "dsa_index_scores": (i32, [pc, pb, P, P, P, i64, P, P]),
            "dsa_topk_workspace_size": (sz, [i32, i32, i32]),
            "dsa_topk": (i32, [P, i64, P, i32, i32, i32, P, P, sz, P, P]),
            "dsa_topk_noalloc": (i32, [P, i64, P, i32, i32, i32, P, P, P]),
            "dsa_topk_force_multipass": (i32, [i32]),
            "dsa_dcp_topk_workspace_size": (sz, [i32, i32, i32]),
            "dsa_dcp_topk": (i32, [P, i64, P, i32, i32, i32, i32, P, P, P, sz, P, P]),
            "sparse_mla_workspace_size": (sz, [i32, i32]),
            "sparse_mla_decode": (i32, [pc, pb, P, P, i32, f32, P, P, P, sz, P, P]),
            "dsa_dcp_sparse_mla_workspace_size": (sz, [i32, i32, i32]),
            "dsa_batch_invariant": (i32, [i32]),
            "dsa_dcp_sparse_mla": (i32, [pc, pb, P, P, i32, i32, f32, P, P, P, P, P, sz, P, P]),
            "dsa_workspace_size": (sz, [pb, i32]),
            "dsa_decode_step": (i32, [pc, pb, P, P, P, i32, f32, P, P, P, i64, P, P, P, sz, P, P]),
            "dsa_decode_step_bf16": (i32, [pc, pb, P, P, P, i32, f32, P, P, P, i64, P, P, P, sz, P, P]),
            "dsa_topk_paged": (i32, [pc, pb, P, i64, i32, P, P, P, sz, P, P]),
            "dsa_index_scores_bf16": (i32, [pc, pb, P, P, P, i64, P, P]),
            "dsa_topk_bf16": (i32, [P, i64, P, i32, i32, i32, P, P, P]),
            "dsa_cache_append": (i32, [pc, pb, P, P, P, P]),
            "dsa_quantize_index_query": (i32, [P, P, i32, P, P, P]),
            "dsa_index_frontend": (i32, [pc, pb, P, i32, P, f32, P, P, P, P, P, P, P, P, P]),
            "dsa_frontend_workspace_size": (sz, [pb, i32]),
            "dsa_decode_step_frontend": (i32, [pc, pb, P, i32, P, f32, P, P, P, P, P, i32, f32, P, P, P, i64, P, P,
                                               P, sz, P, P]),
            "dsa_selftest_wait_timeout": (i32, [i64, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def topk_force_multipass(on: bool) -> bool:
    """Route rows longer than 245,760 tokens through the four-kernel top-k
    (True) or the automatic choice (False); returns the previous setting."""
    return bool(lib().dsa_topk_force_multipass(int(bool(on))))


def kernel_launches() -> int:
    """Kernels libdsa has launched in this process so far."""
    return int(lib().dsa_kernel_launches())


def status_string(code: int) -> str:
    return lib().dsa_status_string(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != OK:
        raise DsaError(code, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors passed to libdsa must be contiguous CUDA tensors")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class PagedCache:
    """One layer's packed paged cache: ``pool`` is a uint8 CUDA tensor
    [num_blocks, row_stride]; offsets locate the latent and index pages."""

    pool: torch.Tensor
    row_stride: int
    latent_off: int
    index_off: int
    key_format: int
    latent_scale: float
    latent_format: int = 0

    def struct(self) -> PagedCacheT:
        return PagedCacheT(_ptr(self.pool), self.row_stride, self.latent_off, self.index_off, BLOCK,
                           int(self.pool.shape[0]), self.key_format, float(self.latent_scale),
                           int(self.latent_format))


@dataclass
class Batch:
    """block_table int32 [batch, max_blocks] and seq_lens int32 [batch] on the GPU."""

    block_table: torch.Tensor
    seq_lens: torch.Tensor
    queries_per_seq: int
    max_seq_len: int

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def rows(self) -> int:
        return self.batch * self.queries_per_seq

    def struct(self) -> BatchT:
        return BatchT(_ptr(self.block_table), _ptr(self.seq_lens), int(self.block_table.shape[1]), self.batch,
                      self.queries_per_seq, int(self.max_seq_len))


def translate_pages(cache: PagedCache, batch: Batch, latent_pages, index_pages, status, stream=None):
    c, b = cache.struct(), batch.struct()
    _check(lib().dsa_translate_pages(ctypes.byref(c), ctypes.byref(b), _ptr(latent_pages), _ptr(index_pages),
                                     _ptr(status), _stream(stream)), "dsa_translate_pages")


def index_scores(cache: PagedCache, batch: Batch, q_index, head_w, scores, status, stream=None):
    c, b = cache.struct(), batch.struct()
    _check(lib().dsa_index_scores(ctypes.byref(c), ctypes.byref(b), _ptr(q_index), _ptr(head_w), _ptr(scores),
                                  int(scores.shape[1]), _ptr(status), _stream(stream)), "dsa_index_scores")


def index_scores_bf16(cache: PagedCache, batch: Batch, q_index, head_w, scores, status, stream=None):
    """Indexer scores rounded to bf16; `scores` holds the bits (int16 or bfloat16 [rows, ld], ld % 8 == 0)."""
    c, b = cache.struct(), batch.struct()
    _check(lib().dsa_index_scores_bf16(ctypes.byref(c), ctypes.byref(b), _ptr(q_index), _ptr(head_w), _ptr(scores),
                                       int(scores.shape[1]), _ptr(status), _stream(stream)), "dsa_index_scores_bf16")


def topk_bf16(scores, row_lens, max_row_len: int, k: int, idx_out, status, stream=None):
    """Top-k over bf16 scores (bits [rows, ld], ld % 8 == 0); no workspace."""
    rows = int(scores.shape[0])
    _check(lib().dsa_topk_bf16(_ptr(scores), int(scores.shape[1]), _ptr(row_lens), rows, int(max_row_len), int(k),
                               _ptr(idx_out), _ptr(status), _stream(stream)), "dsa_topk_bf16")


def topk_workspace_size(rows: int, max_row_len: int, k: int) -> int:
    return int(lib().dsa_topk_workspace_size(rows, max_row_len, k))


def topk(scores, row_lens, max_row_len: int, k: int, idx_out, workspace, status, stream=None):
    rows = int(scores.shape[0])
    _check(lib().dsa_topk(_ptr(scores), int(scores.shape[1]), _ptr(row_lens), rows, int(max_row_len), int(k),
                          _ptr(idx_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _ptr(status), _stream(stream)), "dsa_topk")


def topk_noalloc(scores, row_lens, max_row_len: int, k: int, idx_out, status, stream=None):
    """dsa_topk with the library's built-in scratch: no workspace, no allocation (rows <= 64)."""
    rows = int(scores.shape[0])
    _check(lib().dsa_topk_noalloc(_ptr(scores), int(scores.shape[1]), _ptr(row_lens), rows, int(max_row_len),
                                  int(k), _ptr(idx_out), _ptr(status), _stream(stream)), "dsa_topk_noalloc")


def dcp_topk_workspace_size(rows: int, k: int, shards: int) -> int:
    return int(lib().dsa_dcp_topk_workspace_size(rows, k, shards))


def dcp_topk(scores, row_lens, max_row_len: int, k: int, shards: int, idx_out, workspace, status, stats_out=None,
             stream=None):
    """The decode-context-parallel top-k merge of `shards` token shards (bf16-keyed candidates, global
    selection, resends); stats_out: optional int32 [rows, 3] (words sent, shards that resent, words resent)."""
    rows = int(scores.shape[0])
    _check(lib().dsa_dcp_topk(_ptr(scores), int(scores.shape[1]), _ptr(row_lens), rows, int(max_row_len), int(k),
                              int(shards), _ptr(idx_out), _ptr(stats_out), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "dsa_dcp_topk")


def sparse_mla_workspace_size(rows: int, k: int) -> int:
    return int(lib().sparse_mla_workspace_size(rows, k))


def sparse_mla_decode(cache: PagedCache, batch: Batch, q_mla, idx, sm_scale: float, out, lse, workspace, status,
                      stream=None):
    c, b = cache.struct(), batch.struct()
    _check(lib().sparse_mla_decode(ctypes.byref(c), ctypes.byref(b), _ptr(q_mla), _ptr(idx), int(idx.shape[1]),
                                   float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "sparse_mla_decode")


def batch_invariant(on: bool) -> bool:
    """Switch the process-wide batch-invariant mode (fixed 512-token MLA chunks); returns the previous one."""
    return bool(lib().dsa_batch_invariant(1 if on else 0))


def dcp_sparse_mla_workspace_size(rows: int, k: int, shards: int) -> int:
    return int(lib().dsa_dcp_sparse_mla_workspace_size(rows, k, shards))


def dcp_sparse_mla(cache: PagedCache, batch: Batch, q_mla, idx, shards: int, sm_scale: float, out, lse, workspace,
                   status, part_out=None, part_lse=None, stream=None):
    """Sparse MLA as `shards` token shards would compute it: per-shard partial attention over the selected
    tokens each holds, bf16 partial outputs and fp32 LSEs, merged through their log-sum-exp.  part_out
    (bf16 [shards, rows, 96, 512]) and part_lse (fp32 [shards, rows, 96]) optionally receive the partials."""
    c, b = cache.struct(), batch.struct()
    _check(lib().dsa_dcp_sparse_mla(ctypes.byref(c), ctypes.byref(b), _ptr(q_mla), _ptr(idx), int(idx.shape[1]),
                                    int(shards), float(sm_scale), _ptr(out), _ptr(lse), _ptr(part_out),
                                    _ptr(part_lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _ptr(status), _stream(stream)),
           "dsa_dcp_sparse_mla")


def workspace_size(batch: Batch, k: int) -> int:
    b = batch.struct()
    return int(lib().dsa_workspace_size(ctypes.byref(b), int(k)))


def decode_step(cache: PagedCache, batch: Batch, q_index, head_w, q_mla, k: int, sm_scale: float, out, lse,
                workspace, status, scores_out=None, idx_out=None, stream=None, phys_out=None):
    c, b = cache.struct(), batch.struct()
    ld = int(scores_out.shape[1]) if scores_out is not None else 0
    _check(lib().dsa_decode_step(ctypes.byref(c), ctypes.byref(b), _ptr(q_index), _ptr(head_w), _ptr(q_mla),
                                 int(k), float(sm_scale), _ptr(out), _ptr(lse), _ptr(scores_out), ld,
                                 _ptr(idx_out), _ptr(phys_out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "dsa_decode_step")


def topk_paged(cache: PagedCache, batch: Batch, scores, k: int, idx_out, workspace, status, phys_out=None,
               stream=None):
    """The fused step's top-k on its own (row lengths from the batch), with the
    selected tokens' physical KV rows when phys_out is given."""
    c, b = cache.struct(), batch.struct()
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().dsa_topk_paged(ctypes.byref(c), ctypes.byref(b), _ptr(scores), int(scores.shape[1]), int(k),
                                _ptr(idx_out), _ptr(phys_out), _ptr(workspace), nbytes, _ptr(status),
                                _stream(stream)), "dsa_topk_paged")


def decode_step_bf16(cache: PagedCache, batch: Batch, q_index, head_w, q_mla, k: int, sm_scale: float, out, lse,
                     workspace, status, scores_out=None, idx_out=None, stream=None, phys_out=None):
    """The fused step with bf16 scores between the indexer and the top-k."""
    c, b = cache.struct(), batch.struct()
    ld = int(scores_out.shape[1]) if scores_out is not None else 0
    _check(lib().dsa_decode_step_bf16(ctypes.byref(c), ctypes.byref(b), _ptr(q_index), _ptr(head_w), _ptr(q_mla),
                                      int(k), float(sm_scale), _ptr(out), _ptr(lse), _ptr(scores_out), ld,
                                      _ptr(idx_out), _ptr(phys_out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "dsa_decode_step_bf16")


def cache_append(cache: PagedCache, batch: Batch, new_latent, new_index_key, status, stream=None):
    """Write every sequence's queries_per_seq new tokens (bf16 bits, [rows, 576] and
    [rows, 128]) into their pages."""
    c, b = cache.struct(), batch.struct()
    _check(lib().dsa_cache_append(ctypes.byref(c), ctypes.byref(b), _ptr(new_latent), _ptr(new_index_key),
                                  _ptr(status), _stream(stream)), "dsa_cache_append")


def quantize_index_query(q_bf16, head_w, q_index, head_w_out, stream=None):
    """FP8 indexer query per (row, head), its scale folded into the head weight."""
    rows = int(q_bf16.shape[0])
    _check(lib().dsa_quantize_index_query(_ptr(q_bf16), _ptr(head_w), rows, _ptr(q_index), _ptr(head_w_out),
                                          _stream(stream)), "dsa_quantize_index_query")


def index_frontend(cache: PagedCache, batch: Batch, c_q, gamma, eps: float, w_iq, head_w, new_latent, new_index_key,
                   q_index, head_w_out, status, q_proj=None, stream=None):
    """The fused indexer front end: RMSNorm of c_q (bf16 bits [rows, D]), the
    projection by w_iq (bf16 bits [4096, D]), the FP8 query (q_index [rows, 32,
    128]) with its scale folded into head_w_out, optionally the fp32 projected
    values (q_proj [rows, 4096]), and the new tokens into the cache."""
    c, b = cache.struct(), batch.struct()
    _check(lib().dsa_index_frontend(ctypes.byref(c), ctypes.byref(b), _ptr(c_q), int(c_q.shape[1]), _ptr(gamma),
                                    float(eps), _ptr(w_iq), _ptr(head_w), _ptr(new_latent), _ptr(new_index_key),
                                    _ptr(q_index), _ptr(head_w_out), _ptr(q_proj), _ptr(status), _stream(stream)),
           "dsa_index_frontend")


def frontend_workspace_size(batch: Batch, k: int) -> int:
    b = batch.struct()
    return int(lib().dsa_frontend_workspace_size(ctypes.byref(b), int(k)))


def decode_step_frontend(cache: PagedCache, batch: Batch, c_q, gamma, eps: float, w_iq, head_w, new_latent,
                         new_index_key, q_mla, k: int, sm_scale: float, out, lse, workspace, status, scores_out=None,
                         idx_out=None, stream=None, phys_out=None):
    """The front end, then the fused step over the updated cache (one call)."""
    c, b = cache.struct(), batch.struct()
    ld = int(scores_out.shape[1]) if scores_out is not None else 0
    _check(lib().dsa_decode_step_frontend(ctypes.byref(c), ctypes.byref(b), _ptr(c_q), int(c_q.shape[1]), _ptr(gamma),
                                          float(eps), _ptr(w_iq), _ptr(head_w), _ptr(new_latent),
                                          _ptr(new_index_key), _ptr(q_mla), int(k), float(sm_scale), _ptr(out),
                                          _ptr(lse), _ptr(scores_out), ld, _ptr(idx_out), _ptr(phys_out),
                                          _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(status),
                                          _stream(stream)), "dsa_decode_step_frontend")


def selftest_wait_timeout(limit_ns: int, status, stream=None):
    _check(lib().dsa_selftest_wait_timeout(int(limit_ns), _ptr(status), _stream(stream)),
           "dsa_selftest_wait_timeout")


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned uint8 device buffer (torch's allocator aligns to 512 B)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
