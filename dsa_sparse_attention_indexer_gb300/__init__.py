"""Python binding of libdsa, the GB300 DSA attention-step library.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory, streams and the output buffers.  If the shared
library has not been built, every call raises ``DsaLibraryMissing`` - there is
no fallback.

The function names follow the C ABI in ``include/dsa.h``.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_size_t, c_uint8, c_uint64, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdsa.so")

PAGE_TOKENS = 64
INDEX_HEADS = 32
INDEX_HEAD_DIM = 128
IDXK_TOKEN_BYTES = 132
IDXK_PAGE_BYTES = 8448
IDXK_MXFP4_TOKEN_BYTES = 68
IDXK_MXFP4_PAGE_BYTES = 4352
MLA_HEADS = 64
LATENT_DIM = 512
ROPE_DIM = 64
QK_DIM = 576
KV_TOKEN_BYTES = 656
KV_PAGE_BYTES = 41984
TOPK = 2048
DTYPE_BF16 = 0
DTYPE_F32 = 1

DEVERR_SLOT_RANGE = 1
DEVERR_PAGE_RANGE = 2
DEVERR_INDEX_RANGE = 4
DEVERR_TIMEOUT = 8
DEVERR_FP16_RANGE = 16

ERR = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARGUMENT", 2: "DSA_ERR_ALIGNMENT", 3: "DSA_ERR_UNSUPPORTED",
       4: "DSA_ERR_WORKSPACE_TOO_SMALL", 5: "DSA_ERR_NO_TOPK_SOURCE", 6: "DSA_ERR_CUDA", 7: "DSA_ERR_DEVICE",
       8: "DSA_ERR_SCRATCH_LIMIT"}
NOALLOC_SCRATCH_BYTES = 16 << 20


class DsaLibraryMissing(ImportError):
    pass


class DsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        self.name = ERR.get(code, str(code))
        super().__init__(f"{fn} -> {self.name} ({status_string(code)})")


class DsaScheduleConfig(ctypes.Structure):
    _fields_ = [("indexer_types", POINTER(c_char_p)), ("n_types", c_int32), ("cli_factor", c_int32),
                ("index_topk_pattern", c_char_p), ("index_topk_freq", c_int32), ("index_skip_topk_offset", c_int32)]


class DsaBatch(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("max_pages", c_int32), ("max_seq_len", c_int32),
                ("max_q_len", c_int32), ("total_q", c_int64), ("num_pages", c_int64),
                ("seq_len", c_void_p), ("q_start", c_void_p), ("page_table", c_void_p)]


_lib = None

_SIGS = {
    "dsa_abi_version": (c_int32, []),
    "dsa_status_string": (c_char_p, [c_int32]),
    "dsa_device_status_reset": (c_int32, [c_void_p, c_void_p]),
    "dsa_device_status_read": (c_int32, [c_void_p, c_void_p, POINTER(c_int32)]),
    "dsa_debug_set_wait_limit_ns": (c_int32, [c_uint64]),
    "dsa_index_k_store": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_float,
                                    c_float, c_void_p, c_int64, c_void_p, c_void_p]),
    "dsa_index_k_store_mxfp4": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_float,
                                          c_float, c_void_p, c_int64, c_void_p, c_void_p]),
    "dsa_indexer_topk_mxfp4": (c_int32, [c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_void_p, c_void_p,
                                         c_void_p, c_int32, c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_latent_kv_store_fused": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_float,
                                            c_float, c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_float,
                                            c_void_p, c_int64, c_void_p, c_void_p]),
    "dsa_latent_kv_store": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int64, c_void_p,
                                      c_void_p]),
    "dsa_indexer_topk_workspace_size": (c_int32, [POINTER(DsaBatch), POINTER(c_size_t)]),
    "dsa_indexer_topk": (c_int32, [c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_void_p, c_void_p,
                                   c_void_p, c_int32, c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_indexer_topk_noalloc": (c_int32, [c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_void_p, c_void_p,
                                           c_void_p, c_int32, c_void_p, c_void_p]),
    "dsa_indexer_scores_workspace_size": (c_int32, [POINTER(DsaBatch), POINTER(c_size_t)]),
    "dsa_indexer_scores": (c_int32, [c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_void_p, c_int64,
                                     c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_indexer_scores_cuda_core": (c_int32, [c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_void_p, c_int64,
                                     c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_topk_from_scores_workspace_size": (c_int32, [c_int32, c_int64, POINTER(c_size_t)]),
    "dsa_topk_from_scores": (c_int32, [c_void_p, c_int64, c_void_p, c_int32, c_int64, c_void_p, c_void_p,
                                       c_size_t, c_void_p]),
    "dsa_sparse_mla_workspace_size": (c_int32, [POINTER(DsaBatch), POINTER(c_size_t)]),
    "dsa_sparse_mla_decode": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_float,
                                        c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_sparse_mla_prefill": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, POINTER(DsaBatch), c_float,
                                         c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_parse_indexer_types": (c_int32, [POINTER(c_char_p), c_int32, POINTER(c_uint8)]),
    "dsa_schedule_from_freq": (c_int32, [c_int32, c_int32, c_int32, POINTER(c_uint8)]),
    "dsa_schedule_resolve": (c_int32, [POINTER(DsaScheduleConfig), c_int32, POINTER(c_uint8)]),
    "dsa_topk_share_create": (c_int32, [POINTER(c_void_p)]),
    "dsa_topk_share_destroy": (c_int32, [c_void_p]),
    "dsa_topk_share_reset": (c_int32, [c_void_p]),
    "dsa_topk_share_publish": (c_int32, [c_void_p, c_int32, c_void_p, c_int64]),
    "dsa_topk_share_get": (c_int32, [c_void_p, POINTER(c_void_p), POINTER(c_int64), POINTER(c_int32)]),
    "dsa_mtp_topk_width": (c_int32, [c_int32, c_int32, POINTER(c_int32)]),
    "dsa_mtp_seed_write": (c_int32, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int32, c_void_p, c_void_p]),
    "dsa_topk_share_mtp_begin": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int64, c_int32,
                                           POINTER(c_int32)]),
    "dsa_topk_share_needs_scoring": (c_int32, [c_void_p, POINTER(c_int32)]),
    "dsa_topk_share_mtp_end": (c_int32, [c_void_p]),
    "dsa_cp_topk_merge": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int64, c_void_p, c_void_p, c_void_p,
                                    c_void_p]),
    "dsa_cp_topk_localize": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dsa_cp_attention_merge": (c_int32, [c_void_p, c_void_p, c_int32, c_int64, c_void_p, c_int32, c_void_p,
                                         c_void_p]),
}


def lib():
    """The loaded libdsa (ctypes.CDLL); raises DsaLibraryMissing if not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise DsaLibraryMissing(
                f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def status_string(code: int) -> str:
    return lib().dsa_status_string(code).decode()


def _check(fn: str, code: int):
    if code != 0:
        raise DsaError(fn, code)


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream, device=None):
    """The raw cudaStream_t of `stream` (default: the current stream of
    `device`).  A stream on another device than the call's tensors is refused:
    the kernels would run there with this device's pointers."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != torch.device(device):
        raise ValueError(f"stream is on {stream.device}, the call's tensors on {device}")
    return c_void_p(stream.cuda_stream)


def _call(fn: str, device, *args):
    """Run C entry point `fn` with `device` current, so that the library's
    per-device set-up, its device queries and a default stream all refer to the
    device that holds the call's tensors."""
    with torch.cuda.device(device):
        _check(fn, getattr(lib(), fn)(*args))


def _need(t: torch.Tensor, dtype, name: str, device=None, numel=None):
    """A device argument of the C ABI: a contiguous CUDA tensor of `dtype`, on
    `device` when given, with at least `numel` elements when given.  The
    library reads and writes through raw pointers, so a host tensor, a tensor on
    another GPU or a short buffer is rejected here, before any launch."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
    if device is not None and t.device != torch.device(device):
        raise ValueError(f"{name} is on {t.device}, the call's other tensors on {device}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call needs {numel}")
    return t


def _opt(t, dtype, name: str, device=None, numel=None):
    return None if t is None else _need(t, dtype, name, device, numel)


# ---------------------------------------------------------------------------
class Batch:
    """Owns the device tensors of one batch and the dsa_batch struct over them.

    seq_len int32 [B] and q_start int32 [B+1] (device), page_table int32
    [B, max_pages] (device).  Host bounds default to the tensors' values
    (read once, with a device sync).
    """

    def __init__(self, seq_len, q_start, page_table, num_pages: int, *, max_seq_len=None,
                 max_q_len=None, total_q=None):
        self.seq_len = _need(seq_len, torch.int32, "seq_len")
        self.q_start = _need(q_start, torch.int32, "q_start")
        self.page_table = _need(page_table, torch.int32, "page_table")
        B = seq_len.numel()
        if max_seq_len is None or max_q_len is None or total_q is None:
            sl = seq_len.cpu()
            qs = q_start.cpu()
            max_seq_len = int(sl.max()) if max_seq_len is None else max_seq_len
            max_q_len = int((qs[1:] - qs[:-1]).max()) if max_q_len is None else max_q_len
            total_q = int(qs[-1]) if total_q is None else total_q
        self.c = DsaBatch(B, page_table.shape[1], int(max_seq_len), int(max_q_len), int(total_q),
                          int(num_pages), seq_len.data_ptr(), q_start.data_ptr(), page_table.data_ptr())

    @property
    def total_q(self) -> int:
        return self.c.total_q

    def ref(self):
        return ctypes.byref(self.c)


def _ws_size(fn_name: str, batch: Batch) -> int:
    n = c_size_t(0)
    _check(fn_name, getattr(lib(), fn_name)(batch.ref(), ctypes.byref(n)))
    return n.value


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def new_device_status(device) -> torch.Tensor:
    return torch.zeros(4, dtype=torch.int32, device=device)


def dsa_device_status_read(dev_status: torch.Tensor, stream=None):
    _need(dev_status, torch.int32, "dev_status", numel=4)
    out = (c_int32 * 4)()
    with torch.cuda.device(dev_status.device):
        code = lib().dsa_device_status_read(_ptr(dev_status), _stream(stream, dev_status.device), out)
    if code not in (0, 7):
        _check("dsa_device_status_read", code)
    return list(out)



def dsa_debug_set_wait_limit_ns(ns: int) -> None:
    """Testing hook: limit (ns) of the decode score kernel's pipeline waits for
    later launches, process-wide (2e9 by default; 0 = give up at once)."""
    _check("dsa_debug_set_wait_limit_ns", lib().dsa_debug_set_wait_limit_ns(int(ns)))

def dsa_device_status_reset(dev_status: torch.Tensor, stream=None):
    _need(dev_status, torch.int32, "dev_status", numel=4)
    _call("dsa_device_status_reset", dev_status.device, _ptr(dev_status), _stream(stream, dev_status.device))


# ---------------------------------------------------------------------------
def _store_args(k, pos, slot, idxk_cache, gamma, beta, dev_status):
    _need(k, torch.bfloat16, "k")
    dev, n = k.device, k.shape[0]
    _need(k, torch.bfloat16, "k", dev, n * INDEX_HEAD_DIM)
    _need(pos, torch.int32, "pos", dev, n)
    _need(slot, torch.int64, "slot", dev, n)
    _need(idxk_cache, torch.uint8, "idxk_cache", dev)
    _opt(gamma, torch.float32, "gamma", dev, INDEX_HEAD_DIM)
    _opt(beta, torch.float32, "beta", dev, INDEX_HEAD_DIM)
    _opt(dev_status, torch.int32, "dev_status", dev, 4)
    return n


def dsa_index_k_store(k, pos, slot, idxk_cache, *, gamma=None, beta=None, ln_eps=1e-6,
                      rope_base=10000.0, num_pages=None, dev_status=None, stream=None):
    n = _store_args(k, pos, slot, idxk_cache, gamma, beta, dev_status)
    if num_pages is None:
        num_pages = idxk_cache.numel() // IDXK_PAGE_BYTES
    _call("dsa_index_k_store", k.device,
        _ptr(k), _ptr(pos), _ptr(slot), n, _ptr(gamma), _ptr(beta), ln_eps, rope_base,
        _ptr(idxk_cache), num_pages, _ptr(dev_status), _stream(stream, k.device))


def dsa_index_k_store_mxfp4(k, pos, slot, idxk_cache, *, gamma=None, beta=None, ln_eps=1e-6,
                            rope_base=10000.0, num_pages=None, dev_status=None, stream=None):
    """dsa_index_k_store into an MXFP4 index-K cache (4352-byte pages, 32-byte aligned)."""
    _store_args(k, pos, slot, idxk_cache, gamma, beta, dev_status)
    if num_pages is None:
        num_pages = idxk_cache.numel() // IDXK_MXFP4_PAGE_BYTES
    _call("dsa_index_k_store_mxfp4", k.device,
        _ptr(k), _ptr(pos), _ptr(slot), k.shape[0], _ptr(gamma), _ptr(beta), ln_eps, rope_base,
        _ptr(idxk_cache), num_pages, _ptr(dev_status), _stream(stream, k.device))


def dsa_latent_kv_store_fused(kv_c, k_pe, pos, slot, kv_cache, *, kv_gamma=None, rms_eps=1e-6, rope_base=10000.0,
                              idx_k=None, idxk_cache=None, idx_gamma=None, idx_beta=None, ln_eps=1e-6,
                              num_pages=None, idx_num_pages=None, dev_status=None, stream=None):
    """Latent rows from raw kv_c / k_pe (RMSNorm, RoPE) and, with idx_k, the index keys too."""
    _need(kv_c, torch.bfloat16, "kv_c")
    dev, n = kv_c.device, kv_c.shape[0]
    _need(kv_c, torch.bfloat16, "kv_c", dev, n * LATENT_DIM)
    _need(k_pe, torch.bfloat16, "k_pe", dev, n * ROPE_DIM)
    _need(pos, torch.int32, "pos", dev, n)
    _need(slot, torch.int64, "slot", dev, n)
    _need(kv_cache, torch.uint8, "kv_cache", dev)
    _opt(kv_gamma, torch.float32, "kv_gamma", dev, LATENT_DIM)
    _opt(dev_status, torch.int32, "dev_status", dev, 4)
    if idx_k is not None:
        _need(idx_k, torch.bfloat16, "idx_k", dev, n * INDEX_HEAD_DIM)
        _need(idxk_cache, torch.uint8, "idxk_cache", dev)
        _opt(idx_gamma, torch.float32, "idx_gamma", dev, INDEX_HEAD_DIM)
        _opt(idx_beta, torch.float32, "idx_beta", dev, INDEX_HEAD_DIM)
    if num_pages is None:
        num_pages = kv_cache.numel() // KV_PAGE_BYTES
    if idx_num_pages is None:
        idx_num_pages = 0 if idxk_cache is None else idxk_cache.numel() // IDXK_PAGE_BYTES
    _call("dsa_latent_kv_store_fused", kv_c.device,
        _ptr(kv_c), _ptr(k_pe), _ptr(pos), _ptr(slot), kv_c.shape[0], _ptr(kv_gamma), rms_eps, rope_base,
        _ptr(kv_cache), num_pages, _ptr(idx_k), _ptr(idx_gamma), _ptr(idx_beta), ln_eps, _ptr(idxk_cache),
        idx_num_pages, _ptr(dev_status), _stream(stream, kv_c.device))


def dsa_latent_kv_store(c, rope, slot, kv_cache, *, num_pages=None, dev_status=None, stream=None):
    _need(c, torch.bfloat16, "c")
    dev, n = c.device, c.shape[0]
    _need(c, torch.bfloat16, "c", dev, n * LATENT_DIM)
    _need(rope, torch.bfloat16, "rope", dev, n * ROPE_DIM)
    _need(slot, torch.int64, "slot", dev, n)
    _need(kv_cache, torch.uint8, "kv_cache", dev)
    _opt(dev_status, torch.int32, "dev_status", dev, 4)
    if num_pages is None:
        num_pages = kv_cache.numel() // KV_PAGE_BYTES
    _call("dsa_latent_kv_store", c.device,
        _ptr(c), _ptr(rope), _ptr(slot), c.shape[0], _ptr(kv_cache), num_pages, _ptr(dev_status),
        _stream(stream, c.device))


def _indexer_args(q, w, idxk_cache, batch: Batch) -> int:
    """Checks the indexer's inputs against the batch; returns its query rows T."""
    _need(q, torch.bfloat16, "q")
    T = batch.total_q
    _need(q, torch.bfloat16, "q", q.device, T * INDEX_HEADS * INDEX_HEAD_DIM)
    _need(w, torch.float32, "w", q.device, T * INDEX_HEADS)
    _need(idxk_cache, torch.uint8, "idxk_cache", q.device)
    _need(batch.seq_len, torch.int32, "batch.seq_len", q.device)
    return T


def _ws(ws, nbytes, device):
    """The call's workspace: allocated when not given, else a uint8 CUDA buffer."""
    if ws is None:
        return workspace(nbytes, device)
    return _need(ws, torch.uint8, "ws", device)


def dsa_indexer_topk_workspace_size(batch: Batch) -> int:
    return _ws_size("dsa_indexer_topk_workspace_size", batch)


def dsa_indexer_topk(q, w, idxk_cache, batch: Batch, *, topk=None, topk_scores=None, share=None,
                     layer_id: int = 0, ws=None, dev_status=None, stream=None):
    """Indexer + top-2048.  Returns topk int32 [T, 2048] (allocated if not given)."""
    T = _indexer_args(q, w, idxk_cache, batch)
    if topk is None:
        topk = torch.empty((T, TOPK), dtype=torch.int32, device=q.device)
    _need(topk, torch.int32, "topk", q.device, T * TOPK)
    _opt(topk_scores, torch.float32, "topk_scores", q.device, T * TOPK)
    _opt(dev_status, torch.int32, "dev_status", q.device, 4)
    ws = _ws(ws, dsa_indexer_topk_workspace_size(batch) if ws is None else 0, q.device)
    _call("dsa_indexer_topk", q.device,
        _ptr(q), _ptr(w), _ptr(idxk_cache), batch.ref(), _ptr(topk), _ptr(topk_scores),
        None if share is None else share.handle, layer_id, _ptr(ws), ws.numel(), _ptr(dev_status),
        _stream(stream, q.device))
    return topk


def dsa_indexer_topk_mxfp4(q, w, idxk_cache, batch: Batch, *, topk=None, topk_scores=None, share=None,
                           layer_id: int = 0, ws=None, dev_status=None, stream=None):
    """dsa_indexer_topk over an MXFP4 index-K cache (at most 65535 query rows)."""
    T = _indexer_args(q, w, idxk_cache, batch)
    if topk is None:
        topk = torch.empty((T, TOPK), dtype=torch.int32, device=q.device)
    _need(topk, torch.int32, "topk", q.device, T * TOPK)
    _opt(topk_scores, torch.float32, "topk_scores", q.device, T * TOPK)
    _opt(dev_status, torch.int32, "dev_status", q.device, 4)
    ws = _ws(ws, dsa_indexer_topk_workspace_size(batch) if ws is None else 0, q.device)
    _call("dsa_indexer_topk_mxfp4", q.device,
        _ptr(q), _ptr(w), _ptr(idxk_cache), batch.ref(), _ptr(topk), _ptr(topk_scores),
        None if share is None else share.handle, layer_id, _ptr(ws), ws.numel(), _ptr(dev_status),
        _stream(stream, q.device))
    return topk


def dsa_indexer_topk_noalloc(q, w, idxk_cache, batch: Batch, *, topk=None, topk_scores=None, share=None,
                             layer_id: int = 0, dev_status=None, stream=None):
    """dsa_indexer_topk for decode batches on the library's fixed scratch (no workspace)."""
    T = _indexer_args(q, w, idxk_cache, batch)
    if topk is None:
        topk = torch.empty((T, TOPK), dtype=torch.int32, device=q.device)
    _need(topk, torch.int32, "topk", q.device, T * TOPK)
    _opt(topk_scores, torch.float32, "topk_scores", q.device, T * TOPK)
    _opt(dev_status, torch.int32, "dev_status", q.device, 4)
    _call("dsa_indexer_topk_noalloc", q.device,
        _ptr(q), _ptr(w), _ptr(idxk_cache), batch.ref(), _ptr(topk), _ptr(topk_scores),
        None if share is None else share.handle, layer_id, _ptr(dev_status), _stream(stream, q.device))
    return topk


def dsa_indexer_scores(q, w, idxk_cache, batch: Batch, *, ld=None, scores=None, ws=None,
                       dev_status=None, stream=None):
    """Full fp32 score rows [T, ld] (debug / parity hook)."""
    T = _indexer_args(q, w, idxk_cache, batch)
    ld = batch.c.max_seq_len if ld is None else ld
    if scores is None:
        scores = torch.empty((T, ld), dtype=torch.float32, device=q.device)
    _need(scores, torch.float32, "scores", q.device, T * ld)
    _opt(dev_status, torch.int32, "dev_status", q.device, 4)
    ws = _ws(ws, _ws_size("dsa_indexer_scores_workspace_size", batch) if ws is None else 0, q.device)
    _call("dsa_indexer_scores", q.device,
        _ptr(q), _ptr(w), _ptr(idxk_cache), batch.ref(), _ptr(scores), ld, _ptr(ws), ws.numel(),
        _ptr(dev_status), _stream(stream, q.device))
    return scores


def dsa_indexer_scores_cuda_core(q, w, idxk_cache, batch: Batch, *, ld=None, scores=None, ws=None,
                                 dev_status=None, stream=None):
    """dsa_indexer_scores from the CUDA-core kernel (decode batches; comparison only)."""
    T = _indexer_args(q, w, idxk_cache, batch)
    ld = batch.c.max_seq_len if ld is None else ld
    if scores is None:
        scores = torch.empty((T, ld), dtype=torch.float32, device=q.device)
    _need(scores, torch.float32, "scores", q.device, T * ld)
    _opt(dev_status, torch.int32, "dev_status", q.device, 4)
    ws = _ws(ws, T * (4096 + 128) if ws is None else 0, q.device)
    _call("dsa_indexer_scores_cuda_core", q.device,
        _ptr(q), _ptr(w), _ptr(idxk_cache), batch.ref(), _ptr(scores), ld, _ptr(ws), ws.numel(),
        _ptr(dev_status), _stream(stream, q.device))
    return scores


def dsa_topk_from_scores(scores, valid_len, *, max_len=None, topk=None, stream=None):
    _need(scores, torch.float32, "scores")
    if scores.dim() != 2:
        raise ValueError(f"scores must be [rows, ld], got shape {tuple(scores.shape)}")
    rows, ld = scores.shape
    _need(valid_len, torch.int32, "valid_len", scores.device, rows)
    max_len = ld if max_len is None else max_len
    if topk is None:
        topk = torch.empty((rows, TOPK), dtype=torch.int32, device=scores.device)
    _need(topk, torch.int32, "topk", scores.device, rows * TOPK)
    n = c_size_t(0)
    _check("dsa_topk_from_scores_workspace_size",
           lib().dsa_topk_from_scores_workspace_size(rows, max_len, ctypes.byref(n)))
    ws = workspace(n.value, scores.device)
    _call("dsa_topk_from_scores", scores.device,
        _ptr(scores), ld, _ptr(valid_len), rows, max_len, _ptr(topk), _ptr(ws), ws.numel(), _stream(stream, scores.device))
    return topk


def dsa_sparse_mla_workspace_size(batch: Batch) -> int:
    return _ws_size("dsa_sparse_mla_workspace_size", batch)


def _mla(fn, q, topk, kv_cache, batch, softmax_scale, out, out_dtype, lse, share, ws, dev_status, stream):
    _need(q, torch.bfloat16, "q")
    T = batch.total_q
    dev = q.device
    _need(q, torch.bfloat16, "q", dev, T * MLA_HEADS * QK_DIM)
    _need(kv_cache, torch.uint8, "kv_cache", dev)
    _need(batch.seq_len, torch.int32, "batch.seq_len", dev)
    _opt(topk, torch.int32, "topk", dev, T * TOPK)
    out_t = torch.float32 if out_dtype == DTYPE_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((T, MLA_HEADS, LATENT_DIM), dtype=out_t, device=dev)
    _need(out, out_t, "out", dev, T * MLA_HEADS * LATENT_DIM)
    _opt(lse, torch.float32, "lse", dev, T * MLA_HEADS)
    _opt(dev_status, torch.int32, "dev_status", dev, 4)
    ws = _ws(ws, dsa_sparse_mla_workspace_size(batch) if ws is None else 0, dev)
    _call(fn, dev,
          _ptr(q), _ptr(topk), None if share is None else share.handle, _ptr(kv_cache), batch.ref(),
          softmax_scale, _ptr(out), out_dtype, _ptr(lse), _ptr(ws), ws.numel(), _ptr(dev_status),
          _stream(stream, dev))
    return out


def dsa_sparse_mla_decode(q, topk, kv_cache, batch: Batch, *, softmax_scale=1.0 / 16, out=None,
                          out_dtype=DTYPE_BF16, lse=None, share=None, ws=None, dev_status=None, stream=None):
    return _mla("dsa_sparse_mla_decode", q, topk, kv_cache, batch, softmax_scale, out, out_dtype, lse,
                share, ws, dev_status, stream)


def dsa_sparse_mla_prefill(q, topk, kv_cache, batch: Batch, *, softmax_scale=1.0 / 16, out=None,
                           out_dtype=DTYPE_BF16, lse=None, share=None, ws=None, dev_status=None, stream=None):
    return _mla("dsa_sparse_mla_prefill", q, topk, kv_cache, batch, softmax_scale, out, out_dtype, lse,
                share, ws, dev_status, stream)


# ---------------------------------------------------------------------------
def dsa_parse_indexer_types(types) -> list:
    arr = (c_char_p * len(types))(*[t.encode() for t in types])
    out = (c_uint8 * len(types))()
    _check("dsa_parse_indexer_types", lib().dsa_parse_indexer_types(arr, len(types), out))
    return [bool(v) for v in out]


def dsa_schedule_from_freq(n_layers: int, freq: int, offset: int) -> list:
    out = (c_uint8 * n_layers)()
    _check("dsa_schedule_from_freq", lib().dsa_schedule_from_freq(n_layers, freq, offset, out))
    return [bool(v) for v in out]


def dsa_schedule_resolve(n_layers: int, *, indexer_types=None, cli_factor: int = 1, index_topk_pattern=None,
                         index_topk_freq: int = 1, index_skip_topk_offset=None) -> list:
    """Full (True) / shared (False) per layer from whichever schedule fields a config carries."""
    cfg = DsaScheduleConfig()
    keep = None
    if indexer_types is not None:
        keep = (c_char_p * len(indexer_types))(*[t.encode() for t in indexer_types])
        cfg.indexer_types = ctypes.cast(keep, POINTER(c_char_p))
        cfg.n_types = len(indexer_types)
    cfg.cli_factor = cli_factor
    cfg.index_topk_pattern = None if index_topk_pattern is None else index_topk_pattern.encode()
    cfg.index_topk_freq = index_topk_freq
    cfg.index_skip_topk_offset = -1 if index_skip_topk_offset is None else index_skip_topk_offset
    out = (c_uint8 * n_layers)()
    _check("dsa_schedule_resolve", lib().dsa_schedule_resolve(ctypes.byref(cfg), n_layers, out))
    del keep
    return [bool(v) for v in out]


class TopkShare:
    """The share handle: the last full layer's indices, read by shared layers."""

    def __init__(self):
        h = c_void_p()
        _check("dsa_topk_share_create", lib().dsa_topk_share_create(ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.dsa_topk_share_destroy(self.handle)
            self.handle = None

    def reset(self):
        _check("dsa_topk_share_reset", lib().dsa_topk_share_reset(self.handle))

    def publish(self, layer_id: int, topk: torch.Tensor):
        _need(topk, torch.int32, "topk", numel=topk.shape[0] * TOPK)
        _check("dsa_topk_share_publish",
               lib().dsa_topk_share_publish(self.handle, layer_id, _ptr(topk), topk.shape[0]))

    def get(self):
        """(device pointer, rows, layer_id); raises DsaError(DSA_ERR_NO_TOPK_SOURCE) if empty."""
        p, rows, lid = c_void_p(), c_int64(), c_int32()
        _check("dsa_topk_share_get", lib().dsa_topk_share_get(self.handle, ctypes.byref(p),
                                                               ctypes.byref(rows), ctypes.byref(lid)))
        return p.value, rows.value, lid.value

    # ---- top-k reuse across the draft steps of one MTP iteration
    def mtp_begin(self, enabled: bool = True, eagle_topk: int = 1, keep_carry_seed: bool = False,
                  seed: torch.Tensor = None) -> bool:
        """Start an MTP iteration; returns whether the draft steps reuse top-k.
        seed: optional carried device int32 [rows, 2048] (kept alive by the caller)."""
        if seed is not None:
            _need(seed, torch.int32, "seed")
        on = c_int32()
        rows = 0 if seed is None else seed.shape[0]
        width = 0 if seed is None else seed.shape[1]
        _check("dsa_topk_share_mtp_begin", lib().dsa_topk_share_mtp_begin(
            self.handle, int(bool(enabled)), eagle_topk, int(bool(keep_carry_seed)), _ptr(seed), rows, width,
            ctypes.byref(on)))
        return bool(on.value)

    def needs_scoring(self) -> bool:
        """False while the iteration reuses published indices (skip the indexer)."""
        v = c_int32()
        _check("dsa_topk_share_needs_scoring", lib().dsa_topk_share_needs_scoring(self.handle, ctypes.byref(v)))
        return bool(v.value)

    def mtp_end(self):
        _check("dsa_topk_share_mtp_end", lib().dsa_topk_share_mtp_end(self.handle))

    @contextlib.contextmanager
    def mtp_iteration(self, enabled: bool = True, eagle_topk: int = 1, keep_carry_seed: bool = False,
                      seed: torch.Tensor = None):
        """`with share.mtp_iteration(...) as reuse:` - begin / end around the draft steps."""
        reuse = self.mtp_begin(enabled, eagle_topk, keep_carry_seed, seed)
        try:
            yield reuse
        finally:
            self.mtp_end()


def dsa_mtp_topk_width(index_topk: int = 2048, index_kpool: int = 1) -> int:
    v = c_int32()
    _check("dsa_mtp_topk_width", lib().dsa_mtp_topk_width(index_topk, index_kpool, ctypes.byref(v)))
    return v.value


def dsa_mtp_seed_write(topk, *, src_row=None, n=None, seed=None, width=None, dev_status=None, stream=None):
    """seed[r] = topk[src_row[r]] (2048 int32) followed by -1 tail slots."""
    _need(topk, torch.int32, "topk", numel=topk.shape[0] * TOPK)
    if src_row is not None:
        _need(src_row, torch.int32, "src_row", topk.device)
    if n is None:
        n = topk.shape[0] if src_row is None else src_row.shape[0]
    if width is None:
        width = dsa_mtp_topk_width() if seed is None else seed.shape[1]
    if seed is None:
        seed = torch.empty((n, width), dtype=torch.int32, device=topk.device)
    _need(seed, torch.int32, "seed", topk.device, n * width)
    _opt(dev_status, torch.int32, "dev_status", topk.device, 4)
    _call("dsa_mtp_seed_write", topk.device,
        _ptr(topk), topk.shape[0], _ptr(src_row), n, _ptr(seed), width, _ptr(dev_status), _stream(stream, topk.device))
    return seed


def index_cache_scale_view(idxk_cache: torch.Tensor) -> torch.Tensor:
    """fp32 [num_pages, 64] view of the per-token scales inside an index-K cache."""
    pages = idxk_cache.view(-1, IDXK_PAGE_BYTES)
    return pages[:, PAGE_TOKENS * INDEX_HEAD_DIM:].view(torch.float32)


# ---------------------------------------------------------------------------
# Context-parallel split of long requests over the ranks of a process group
# ("GLM-5.3 推理全链路(十一)", 两个框架的对照; "Accelerating GLM-5.3-Flash on H200",
# prefill 的重点是少搬一次、少等一次).  See dsa.h for the steps.
CP_MAX_RANKS = 8


def dsa_cp_topk_merge(cand_pos, cand_scores, pos_offset, *, topk=None, topk_scores=None, dev_status=None,
                      stream=None):
    """Global top-2048 from every rank's list: cand_pos / cand_scores [G, rows, 2048],
    pos_offset int64 [G, rows].  Returns topk int32 [rows, 2048]."""
    _need(cand_pos, torch.int32, "cand_pos")
    if cand_pos.dim() != 3 or cand_pos.shape[2] != TOPK:
        raise ValueError(f"cand_pos must be [G, rows, {TOPK}], got {tuple(cand_pos.shape)}")
    G, rows = cand_pos.shape[0], cand_pos.shape[1]
    dev = cand_pos.device
    _need(cand_scores, torch.float32, "cand_scores", dev, G * rows * TOPK)
    _need(pos_offset, torch.int64, "pos_offset", dev, G * rows)
    if topk is None:
        topk = torch.empty((rows, TOPK), dtype=torch.int32, device=dev)
    _need(topk, torch.int32, "topk", dev, rows * TOPK)
    _opt(topk_scores, torch.float32, "topk_scores", dev, rows * TOPK)
    _opt(dev_status, torch.int32, "dev_status", dev, 4)
    _call("dsa_cp_topk_merge", dev, _ptr(cand_pos), _ptr(cand_scores), _ptr(pos_offset), G, rows, _ptr(topk),
          _ptr(topk_scores), _ptr(dev_status), _stream(stream, dev))
    return topk


def dsa_cp_topk_localize(topk, slice_start, slice_len, *, local_topk=None, stream=None):
    """This rank's share of a global top-k list, in local positions, compacted."""
    _need(topk, torch.int32, "topk")
    rows, dev = topk.shape[0], topk.device
    _need(topk, torch.int32, "topk", dev, rows * TOPK)
    _need(slice_start, torch.int64, "slice_start", dev, rows)
    _need(slice_len, torch.int64, "slice_len", dev, rows)
    if local_topk is None:
        local_topk = torch.empty((rows, TOPK), dtype=torch.int32, device=dev)
    _need(local_topk, torch.int32, "local_topk", dev, rows * TOPK)
    _call("dsa_cp_topk_localize", dev, _ptr(topk), rows, _ptr(slice_start), _ptr(slice_len), _ptr(local_topk),
          _stream(stream, dev))
    return local_topk


def dsa_cp_attention_merge(o_parts, lse_parts, *, out=None, out_dtype=DTYPE_BF16, lse=None, stream=None):
    """Attention over the union of the ranks' selected positions from their
    parts: o_parts fp32 [G, rows, 64, 512], lse_parts fp32 [G, rows, 64]."""
    _need(o_parts, torch.float32, "o_parts")
    if o_parts.dim() != 4 or tuple(o_parts.shape[2:]) != (MLA_HEADS, LATENT_DIM):
        raise ValueError(f"o_parts must be [G, rows, 64, 512], got {tuple(o_parts.shape)}")
    G, rows, dev = o_parts.shape[0], o_parts.shape[1], o_parts.device
    _need(lse_parts, torch.float32, "lse_parts", dev, G * rows * MLA_HEADS)
    out_t = torch.float32 if out_dtype == DTYPE_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((rows, MLA_HEADS, LATENT_DIM), dtype=out_t, device=dev)
    _need(out, out_t, "out", dev, rows * MLA_HEADS * LATENT_DIM)
    _opt(lse, torch.float32, "lse", dev, rows * MLA_HEADS)
    _call("dsa_cp_attention_merge", dev, _ptr(o_parts), _ptr(lse_parts), G, rows, _ptr(out), out_dtype, _ptr(lse),
          _stream(stream, dev))
    return out


class LibraryOps:
    """The per-rank steps of the context-parallel split, as library calls."""

    def indexer_topk(self, q, w, idxk_cache, batch, ws=None, dev_status=None, stream=None):
        T = batch.total_q
        topk = torch.empty((T, TOPK), dtype=torch.int32, device=q.device)
        scores = torch.empty((T, TOPK), dtype=torch.float32, device=q.device)
        dsa_indexer_topk(q, w, idxk_cache, batch, topk=topk, topk_scores=scores, ws=ws, dev_status=dev_status,
                         stream=stream)
        return topk, scores

    def topk_merge(self, cand_pos, cand_scores, pos_offset, dev_status=None, stream=None):
        return dsa_cp_topk_merge(cand_pos, cand_scores, pos_offset, dev_status=dev_status, stream=stream)

    def topk_localize(self, topk, slice_start, slice_len, stream=None):
        return dsa_cp_topk_localize(topk, slice_start, slice_len, stream=stream)

    def sparse_mla(self, q, local_topk, kv_cache, batch, softmax_scale, ws=None, dev_status=None, stream=None):
        T = batch.total_q
        lse = torch.empty((T, MLA_HEADS), dtype=torch.float32, device=q.device)
        out = dsa_sparse_mla_decode(q, local_topk, kv_cache, batch, softmax_scale=softmax_scale, out_dtype=DTYPE_F32,
                                    lse=lse, ws=ws, dev_status=dev_status, stream=stream)
        return out, lse

    def attention_merge(self, o_parts, lse_parts, out_dtype, stream=None):
        T = o_parts.shape[1]
        lse = torch.empty((T, MLA_HEADS), dtype=torch.float32, device=o_parts.device)
        out = dsa_cp_attention_merge(o_parts, lse_parts, out_dtype=out_dtype, lse=lse, stream=stream)
        return out, lse


def _gather_ranks(t, group):
    """[G, *t.shape]: every rank's t, in rank order (the exchange step)."""
    import torch.distributed as dist
    G = dist.get_world_size(group)
    if dist.get_backend(group) == "nccl":
        out = torch.empty((G, *t.shape), dtype=t.dtype, device=t.device)
        dist.all_gather_into_tensor(out, t.contiguous(), group=group)
        return out
    parts = [torch.empty_like(t) for _ in range(G)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


class ContextParallel:
    """One layer's indexer and sparse MLA for requests whose positions are cut
    into disjoint slices, one per rank of `group` (at most 8 ranks).  This rank
    holds its slice of every request in its own caches, described by `batch`
    as requests of seq_len = slice length with local positions; slice_start
    (int64 [rows], device) gives the global position of each row's local
    position 0, slice_len the slice's length.  Every slice must be longer than
    2048 tokens.  Two exchanges per layer: at most 2048 (score, position) pairs
    per row and rank after the indexer, one [64, 512] fp32 part and its
    log-sum-exp per row and rank after sparse MLA.

    `ops` performs the per-rank steps; it defaults to the library's calls."""

    def __init__(self, group=None, ops=None, gather=None):
        import torch.distributed as dist
        self.group = group
        self.world = dist.get_world_size(group)
        if self.world > CP_MAX_RANKS:
            raise ValueError(f"at most {CP_MAX_RANKS} ranks, the group has {self.world}")
        self.ops = ops if ops is not None else LibraryOps()
        self._gather = gather if gather is not None else (lambda t: _gather_ranks(t, group))

    def indexer_topk(self, q, w, idxk_cache, batch, slice_start, *, share=None, layer_id=0, ws=None,
                     dev_status=None, stream=None):
        """The global top-2048 of every row (global positions, ascending)."""
        local, scores = self.ops.indexer_topk(q, w, idxk_cache, batch, ws=ws, dev_status=dev_status, stream=stream)
        cand_pos = self._gather(local)
        cand_scores = self._gather(scores)
        offsets = self._gather(slice_start)
        topk = self.ops.topk_merge(cand_pos, cand_scores, offsets, dev_status=dev_status, stream=stream)
        if share is not None:
            share.publish(layer_id, topk)
        return topk

    def sparse_mla(self, q, topk, kv_cache, batch, slice_start, slice_len, *, softmax_scale=1.0 / 16,
                   out_dtype=DTYPE_BF16, ws=None, dev_status=None, stream=None):
        """Attention of every row over its global top-2048; returns (out, lse)."""
        local = self.ops.topk_localize(topk, slice_start, slice_len, stream=stream)
        o, lse = self.ops.sparse_mla(q, local, kv_cache, batch, softmax_scale, ws=ws, dev_status=dev_status,
                                     stream=stream)
        return self.ops.attention_merge(self._gather(o), self._gather(lse), out_dtype, stream=stream)
