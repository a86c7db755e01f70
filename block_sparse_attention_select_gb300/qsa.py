"""Thin ctypes binding of libqsa.so (declared in include/qsa.h).

Same entry points as the C ABI; this module only checks tensor dtypes and
devices, passes raw pointers and the current CUDA stream, and turns a status
code into an exception.  Every step of the indexer runs in the library's
kernels.  There is no fallback: if the library is missing, loading raises.

PyTorch supplies device memory (outputs and workspace, when the caller does
not pass them) and streams.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qsa.h")

QSA_OK = 0
QSA_ERR_INVALID_ARG = 1
QSA_ERR_UNSUPPORTED = 2
QSA_ERR_WORKSPACE = 3
QSA_ERR_LAUNCH = 4
QSA_ERR_BAD_PAGE = 5
QSA_ERR_TIMEOUT = 6
QSA_ERR_CUDA = 7
QSA_ERR_NO_DEVICE = 8
QSA_ERR_STATIC_LIMIT = 9

QSA_CFG_PATH = 1
QSA_CFG_WAIT_LIMIT_NS = 2
QSA_CFG_KERNEL_TIMING = 3
QSA_CFG_OVERLAP = 4
QSA_CFG_CLUSTER = 5
KERNEL_KINDS = ["plan", "score_logits", "score_sample", "score_filter", "score_blocks",
                "select_dense", "select_thresh", "select_cand", "unused8", "pad"]
PATH_AUTO, PATH_DENSE, PATH_FILTER = 0, 1, 2


def _max_k_from_header() -> int:
    with open(HEADER) as f:
        m = re.search(r"#define\s+QSA_MAX_K\s+(\d+)", f.read())
    return int(m.group(1))


QSA_MAX_K = _max_k_from_header()


class QSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class PagedKeysC(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("page_positions", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("num_reqs", ctypes.c_int32),
                ("max_pages_per_req", ctypes.c_int32)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libqsa.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"libqsa.so not built at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    kp = ctypes.POINTER(PagedKeysC)
    lib.qsa_workspace_bytes.restype = sz
    lib.qsa_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.qsa_index_score.restype = ctypes.c_int
    lib.qsa_index_score.argtypes = [vp, vp, i32, i32, kp, vp, vp, vp, i64, vp, sz, vp]
    lib.qsa_topk_exact.restype = ctypes.c_int
    lib.qsa_topk_exact.argtypes = [vp, i64, i32, vp, i32, vp, vp, vp, sz, vp]
    lib.qsa_select_paged_tokens.restype = ctypes.c_int
    lib.qsa_select_paged_tokens.argtypes = [vp, vp, i32, i32, kp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.qsa_get_device_status.restype = ctypes.c_int
    lib.qsa_get_device_status.argtypes = [vp]
    lib.qsa_status_string.restype = ctypes.c_char_p
    lib.qsa_status_string.argtypes = [ctypes.c_int]
    lib.qsa_set_config.restype = ctypes.c_int
    lib.qsa_set_config.argtypes = [i32, i64]
    lib.qsa_last_launch_count.restype = i32
    lib.qsa_last_launch_count.argtypes = []
    lib.qsa_last_cluster_size.restype = i32
    lib.qsa_last_cluster_size.argtypes = []
    lib.qsa_select_paged_tokens_noalloc.restype = ctypes.c_int
    lib.qsa_select_paged_tokens_noalloc.argtypes = [vp, vp, i32, i32, kp, vp, vp, i32, vp, vp, vp]
    lib.qsa_kernel_times.restype = ctypes.c_int
    lib.qsa_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32), i32]
    lib.qsa_sparse_attention.restype = ctypes.c_int
    lib.qsa_sparse_attention.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, i32, vp, i32, i32, vp, vp, vp, i32,
                                         ctypes.c_float, vp, vp]
    lib.qsa_rope_table.restype = ctypes.c_int
    lib.qsa_rope_table.argtypes = [vp, i32, i32, ctypes.c_double, vp]
    lib.qsa_block_select_workspace_bytes.restype = sz
    lib.qsa_block_select_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.qsa_block_select.restype = ctypes.c_int
    lib.qsa_block_select.argtypes = [vp, i32, i32, vp, i32, vp, i32, i32, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.qsa_index_key_produce.restype = ctypes.c_int
    lib.qsa_index_key_produce.argtypes = [vp, vp, i32, vp, vp, i32, vp, ctypes.c_float, vp, i32, i32, i32,
                                          kp, vp]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().qsa_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != QSA_OK:
        raise QSAError(status, where)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class PagedKeys:
    """Paged index-key cache: k_cache fp16 [num_pages, P, 128], block_table int32 [B, max_pages]."""

    def __init__(self, k_cache: torch.Tensor, block_table: torch.Tensor):
        _need(k_cache, torch.float16, "k_cache")
        _need(block_table, torch.int32, "block_table")
        assert k_cache.dim() == 3 and block_table.dim() == 2
        self.k_cache = k_cache
        self.block_table = block_table
        self.c = PagedKeysC(k_cache.data_ptr(), k_cache.shape[0], k_cache.shape[1],
                            k_cache.shape[2], block_table.data_ptr(), block_table.shape[0],
                            block_table.shape[1])

    @property
    def max_len(self) -> int:
        return int(self.block_table.shape[1]) * int(self.k_cache.shape[1])


def workspace_bytes(rows: int, row_capacity: int, k: int, flags: int = 0) -> int:
    return int(load().qsa_workspace_bytes(int(rows), int(row_capacity), int(k), int(flags)))


def alloc_workspace(rows: int, row_capacity: int, k: int, device=None) -> torch.Tensor:
    n = workspace_bytes(rows, row_capacity, k)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def index_score(q, w, keys: PagedKeys, row_req, row_visible, logits, ws=None, stream=None):
    """logits [R, ld] fp32 <- scores (-inf past each row's visible length)."""
    _need(q, torch.float16, "q"), _need(w, torch.float32, "w"), _need(logits, torch.float32, "logits")
    _need(row_req, torch.int32, "row_req"), _need(row_visible, torch.int32, "row_visible")
    R, H = int(q.shape[0]), int(q.shape[1])
    if ws is None:
        ws = alloc_workspace(R, 1, 1, q.device)
    st = load().qsa_index_score(_ptr(q), _ptr(w), R, H, ctypes.byref(keys.c), _ptr(row_req),
                                _ptr(row_visible), _ptr(logits), int(logits.shape[1]), _ptr(ws),
                                ws.numel(), _stream(stream))
    _check(st, "qsa_index_score")
    return logits


def topk_exact(logits, row_visible, k: int, out_idx=None, out_val=None, ws=None, stream=None,
               with_values: bool = True):
    _need(logits, torch.float32, "logits"), _need(row_visible, torch.int32, "row_visible")
    R = int(logits.shape[0])
    if out_idx is None:
        out_idx = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    if out_val is None and with_values:
        out_val = torch.empty((R, k), dtype=torch.float32, device=logits.device)
    st = load().qsa_topk_exact(_ptr(logits), int(logits.stride(0)), R, _ptr(row_visible), int(k),
                               _ptr(out_idx), _ptr(out_val), _ptr(ws),
                               0 if ws is None else ws.numel(), _stream(stream))
    _check(st, "qsa_topk_exact")
    return out_idx, out_val


def select_paged_tokens(q, w, keys: PagedKeys, row_req, row_visible, k: int, out_idx=None,
                        out_val=None, ws=None, stream=None, with_values: bool = True):
    """Exact top-k positions per row: (out_idx int32 [R,k], out_val fp32 [R,k] or None)."""
    _need(q, torch.float16, "q"), _need(w, torch.float32, "w")
    _need(row_req, torch.int32, "row_req"), _need(row_visible, torch.int32, "row_visible")
    R, H = int(q.shape[0]), int(q.shape[1])
    if out_idx is None:
        out_idx = torch.empty((R, k), dtype=torch.int32, device=q.device)
    if out_val is None and with_values:
        out_val = torch.empty((R, k), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(R, keys.max_len, k, q.device)
    st = load().qsa_select_paged_tokens(_ptr(q), _ptr(w), R, H, ctypes.byref(keys.c),
                                        _ptr(row_req), _ptr(row_visible), int(k), _ptr(out_idx),
                                        _ptr(out_val), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "qsa_select_paged_tokens")
    return out_idx, out_val


def select_paged_tokens_noalloc(q, w, keys: PagedKeys, row_req, row_visible, k: int, out_idx,
                                out_val=None, stream=None):
    """select_paged_tokens without a workspace: the library's own static scratch
    buffer is used (for callers that cannot allocate device memory).  Outputs
    must be passed in; calls on one device must not overlap."""
    _need(q, torch.float16, "q"), _need(w, torch.float32, "w")
    _need(row_req, torch.int32, "row_req"), _need(row_visible, torch.int32, "row_visible")
    _need(out_idx, torch.int32, "out_idx")
    R, H = int(q.shape[0]), int(q.shape[1])
    st = load().qsa_select_paged_tokens_noalloc(_ptr(q), _ptr(w), R, H, ctypes.byref(keys.c),
                                                _ptr(row_req), _ptr(row_visible), int(k),
                                                _ptr(out_idx), _ptr(out_val), _stream(stream))
    _check(st, "qsa_select_paged_tokens_noalloc")
    return out_idx, out_val


def rope_table(n_blocks: int, rope_dim: int = 64, theta: float = 10000.0, device=None, stream=None):
    """cos / sin rows of the block-start positions 4i, i < n_blocks: FP32 [n_blocks, rope_dim]."""
    t = torch.empty((max(int(n_blocks), 1), max(int(rope_dim), 8)), dtype=torch.float32,
                    device=device or "cuda")
    _check(load().qsa_rope_table(_ptr(t), int(n_blocks), int(rope_dim), float(theta), _stream(stream)),
           "qsa_rope_table")
    return t


def index_key_produce(x, seq_start, pos_start, max_tokens: int, norm_weight, rope_tab, keys: PagedKeys,
                      pool_logit=None, eps: float = 1e-6, rope_dim: int = 64, window: int = 4, stream=None):
    """Pool, RMS-normalise, rotate and store the index key of every block the new
    tokens complete (x FP16 [T, 128]; seq_start int32 [B + 1]; pos_start int32
    [B]) into keys.k_cache, in place."""
    _need(x, torch.float16, "x"), _need(seq_start, torch.int32, "seq_start")
    _need(pos_start, torch.int32, "pos_start"), _need(norm_weight, torch.float32, "norm_weight")
    if pool_logit is not None:
        _need(pool_logit, torch.float32, "pool_logit")
    if rope_tab is not None:
        _need(rope_tab, torch.float32, "rope_tab")
    rope_blocks = int(rope_tab.shape[0]) if rope_tab is not None else 0
    st = load().qsa_index_key_produce(_ptr(x), _ptr(pool_logit), int(pos_start.shape[0]), _ptr(seq_start),
                                      _ptr(pos_start), int(max_tokens), _ptr(norm_weight), float(eps),
                                      _ptr(rope_tab), rope_blocks, int(rope_dim), int(window),
                                      ctypes.byref(keys.c), _stream(stream))
    _check(st, "qsa_index_key_produce")


def sparse_attention(q, k_cache, v_cache, block_table, row_req, row_token, sel, scale=None, out=None,
                     stream=None):
    """Each row attends the raw tokens of its selected index positions (and its
    unfinished block): q FP16 [R, hq, 256]; caches FP16 [pages, page_tokens, hkv,
    256]; block_table int32 [B, max_pages]; sel int32 [R, k].  Returns FP32
    [R, hq, 256]."""
    _need(q, torch.float16, "q"), _need(k_cache, torch.float16, "k_cache")
    _need(v_cache, torch.float16, "v_cache"), _need(block_table, torch.int32, "block_table")
    _need(row_req, torch.int32, "row_req"), _need(row_token, torch.int32, "row_token")
    _need(sel, torch.int32, "sel")
    R, hq, D = (int(x) for x in q.shape)
    npg, pt, hkv = (int(x) for x in k_cache.shape[:3])
    if out is None:
        out = torch.empty((R, hq, D), dtype=torch.float32, device=q.device)
    scale = 1.0 / (D ** 0.5) if scale is None else float(scale)
    st = load().qsa_sparse_attention(_ptr(q), R, hq, _ptr(k_cache), _ptr(v_cache), npg, pt, hkv, D,
                                     _ptr(block_table), int(block_table.shape[0]), int(block_table.shape[1]),
                                     _ptr(row_req), _ptr(row_token), _ptr(sel), int(sel.shape[1]), scale,
                                     _ptr(out), _stream(stream))
    _check(st, "qsa_sparse_attention")
    return out


def block_select(q, k_cache, block_table, row_req, row_token, k: int, out_idx=None, out_val=None, ws=None,
                 stream=None, with_values: bool = True):
    """Block scorer (the M3-style second workload): top-k 128-token blocks per
    (row, head) by the maximum query-key dot product over each block's visible
    tokens.  q FP16 [R, H, 128]; k_cache FP16 [pages, 128, H, 128]; block_table
    int32 [B, max_blocks]; row_req, row_token int32 [R].  Returns (int32 [R, H,
    k], FP32 [R, H, k] or None)."""
    _need(q, torch.float16, "q"), _need(k_cache, torch.float16, "k_cache")
    _need(block_table, torch.int32, "block_table"), _need(row_req, torch.int32, "row_req")
    _need(row_token, torch.int32, "row_token")
    R, H = int(q.shape[0]), int(q.shape[1])
    nb, mb = int(block_table.shape[0]), int(block_table.shape[1])
    if out_idx is None:
        out_idx = torch.empty((R, H, k), dtype=torch.int32, device=q.device)
    if out_val is None and with_values:
        out_val = torch.empty((R, H, k), dtype=torch.float32, device=q.device)
    if ws is None:
        n = int(load().qsa_block_select_workspace_bytes(R, H, mb, int(k)))
        ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    st = load().qsa_block_select(_ptr(q), R, H, _ptr(k_cache), int(k_cache.shape[0]), _ptr(block_table), nb, mb,
                                 _ptr(row_req), _ptr(row_token), int(k), _ptr(out_idx), _ptr(out_val), _ptr(ws),
                                 ws.numel(), _stream(stream))
    _check(st, "qsa_block_select")
    return out_idx, out_val


def get_device_status(stream=None) -> int:
    return int(load().qsa_get_device_status(_stream(stream)))


def set_config(key: int, value: int):
    _check(load().qsa_set_config(int(key), int(value)), "qsa_set_config")


def last_launch_count() -> int:
    return int(load().qsa_last_launch_count())


def last_cluster_size() -> int:
    return int(load().qsa_last_cluster_size())


def kernel_times():
    """{kind: (total ms, launches)} of the launches timed since the last call."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int32 * n)()
    _check(load().qsa_kernel_times(ms, cnt, n), "qsa_kernel_times")
    return {KERNEL_KINDS[i]: (ms[i], cnt[i]) for i in range(n) if cnt[i]}
