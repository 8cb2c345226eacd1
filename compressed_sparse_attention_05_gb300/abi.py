"""ctypes binding of libcsa2.so: the entry points of include/csa2.h, same names.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and the
current stream); sizes and pointers are handed to the C ABI unchanged.  If the
library is missing, loading raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa2.so")

CSA2_OK = 0
CSA2_F32, CSA2_BF16 = 0, 1
CSA2_KV_MXFP4, CSA2_KV_FP8 = 0, 1
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
STATUS_BAD_PAGE, STATUS_BAD_INDEX, STATUS_BAD_COUNT = 1, 2, 4

ERRORS = {1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED", 3: "CSA2_ERR_CUDA",
          4: "CSA2_ERR_WORKSPACE", 5: "CSA2_ERR_DEVICE_DATA"}


class Csa2Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Dims(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("B", "Tq", "d", "r", "Hq", "Hi", "Di", "idx_dtype", "K", "W",
                                        "max_pages", "n_pool_blocks", "pool_block", "swa_cap", "kv_format")]


class Cache(C.Structure):
    _fields_ = [("kv_codes", C.c_void_p), ("kv_scales", C.c_void_p), ("idx_k", C.c_void_p),
                ("page_table", C.c_void_p), ("n_entries", C.c_void_p), ("n_pages", C.c_int64)]


class Window(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("pos0", C.c_void_p)]


class LayerArgs(C.Structure):
    _fields_ = [
        ("mode", C.c_int32), ("hierarchical", C.c_int32), ("dims", Dims), ("cache", Cache),
        ("window", Window), ("q_pos", C.c_void_p), ("max_entries", C.c_int32),
        ("hidden", C.c_void_p), ("T", C.c_int32), ("H", C.c_int32), ("W_c", C.c_void_p),
        ("W_idx", C.c_void_p), ("gamma", C.c_void_p), ("eps", C.c_float), ("rope_base", C.c_float),
        ("first_entry", C.c_void_p), ("swa_new", C.c_void_p), ("idx_q", C.c_void_p),
        ("idx_w", C.c_void_p), ("Q", C.c_void_p), ("softmax_scale", C.c_float),
        ("idx_in", C.c_void_p), ("cnt_in", C.c_void_p), ("idx_out", C.c_void_p),
        ("cnt_out", C.c_void_p), ("pool", C.c_void_p), ("pool_cnt", C.c_void_p),
        ("O", C.c_void_p), ("lse", C.c_void_p),
    ]


_P, _I32, _I64, _F, _SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t

# name -> (restype, argtypes), in the order of include/csa2.h
SIGNATURES = {
    "csa2_abi_version": (C.c_int, []),
    "csa2_launch_count": (C.c_uint64, []),
    "csa2_last_error": (C.c_char_p, []),
    "csa2_get_status": (C.c_int, [C.POINTER(C.c_uint32), _P]),
    "csa2_pack_mxfp4_f32": (C.c_int, [_P, _I64, _I32, _P, _P, _P]),
    "csa2_unpack_mxfp4_bf16": (C.c_int, [_P, _P, _I64, _I32, _P, _P]),
    "csa2_pack_swa_fp8": (C.c_int, [_P, _I64, _I32, _P, _P, _P]),
    "csa2_norm_rope_pack": (C.c_int, [_P, _I32, _I32, _I32, _I32, _P, _F, _F, _P, _P, _P, _I32, _I64,
                                      _P, _P, _P]),
    "csa2_norm_rope_pack_fp8": (C.c_int, [_P, _I32, _I32, _I32, _I32, _P, _F, _F, _P, _P, _P, _I32, _I64,
                                          _P, _P, _P]),
    "csa2_compress_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "csa2_compress_pack": (C.c_int, [_P, _I32, _I32, _I32, _P, _P, _F, _F, _P, _P, C.POINTER(Dims),
                                     C.POINTER(Cache), _P, _SZ, _P]),
    "csa2_compress_layers_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "csa2_compress_layers": (C.c_int, [_P, _I32, _I32, _I32, _I32, _P, _I32, _P, _F, _F, _P, C.POINTER(Dims),
                                       C.POINTER(Cache), _P, _SZ, _P]),
    "csa2_swa_replay_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "csa2_swa_replay": (C.c_int, [_P, _I32, _I32, _I32, _P, _P, _F, _F, _P, C.POINTER(Dims), C.POINTER(Window),
                                  _P, _SZ, _P]),
    "csa2_index_scores": (C.c_int, [C.POINTER(Dims), C.POINTER(Cache), _P, _P, _P, _P, _I64, _P, _I64, _P]),
    "csa2_topk_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "csa2_topk_f32": (C.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "csa2_block_pool_f32": (C.c_int, [_P, _I64, _I64, _P, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "csa2_index_topk_workspace_size": (_SZ, [C.POINTER(Dims), _I32]),
    "csa2_index_topk": (C.c_int, [C.POINTER(Dims), C.POINTER(Cache), _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _I32, _P, _SZ, _P]),
    "csa2_index_topk_noalloc_capacity": (_SZ, []),
    "csa2_index_topk_noalloc": (C.c_int, [C.POINTER(Dims), C.POINTER(Cache), _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _I32, _P]),
    "csa2_sparse_attn": (C.c_int, [C.POINTER(Dims), C.POINTER(Cache), C.POINTER(Window), _P, _P, _P, _P,
                                   _F, _P, _P, _P]),
    "csa2_layer_workspace_size": (_SZ, [C.POINTER(LayerArgs)]),
    "csa2_layer": (C.c_int, [C.POINTER(LayerArgs), _P, _SZ, _P]),
}

_lib = None


def lib():
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m compressed_sparse_attention_05_gb300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(rc: int):
    if rc != CSA2_OK:
        raise Csa2Error(rc, lib().csa2_last_error().decode())


def ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def stream_handle(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def bits16(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensors travel as their 16-bit patterns."""
    assert t.dtype == torch.bfloat16
    return t


# ---- entry points ---------------------------------------------------------------

def csa2_abi_version() -> int:
    return lib().csa2_abi_version()


def csa2_launch_count() -> int:
    return lib().csa2_launch_count()


def csa2_get_status(stream=None) -> int:
    bits = C.c_uint32(0)
    _check(lib().csa2_get_status(C.byref(bits), stream_handle(stream)))
    return bits.value


def csa2_pack_mxfp4_f32(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None):
    n, d = x.shape
    _check(lib().csa2_pack_mxfp4_f32(ptr(x), n, d, ptr(codes), ptr(scales), stream_handle(stream)))


def csa2_unpack_mxfp4_bf16(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None):
    n, d = out.shape
    _check(lib().csa2_unpack_mxfp4_bf16(ptr(codes), ptr(scales), n, d, ptr(out), stream_handle(stream)))


def csa2_pack_swa_fp8(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None):
    n, d = x.shape
    _check(lib().csa2_pack_swa_fp8(ptr(x), n, d, ptr(codes), ptr(scales), stream_handle(stream)))


def csa2_norm_rope_pack(latent, r, gamma, eps, rope_base, first_entry, n_rows, page_table, n_pages,
                        kv_codes, kv_scales, stream=None):
    B, n_max, d = latent.shape
    _check(lib().csa2_norm_rope_pack(ptr(latent), B, n_max, d, r, ptr(gamma), eps, rope_base,
                                     ptr(first_entry), ptr(n_rows), ptr(page_table), page_table.shape[1],
                                     n_pages, ptr(kv_codes), ptr(kv_scales), stream_handle(stream)))


def csa2_norm_rope_pack_fp8(latent, r, gamma, eps, rope_base, first_entry, n_rows, page_table, n_pages,
                            kv_codes, kv_scales, stream=None):
    B, n_max, d = latent.shape
    _check(lib().csa2_norm_rope_pack_fp8(ptr(latent), B, n_max, d, r, ptr(gamma), eps, rope_base,
                                         ptr(first_entry), ptr(n_rows), ptr(page_table), page_table.shape[1],
                                         n_pages, ptr(kv_codes), ptr(kv_scales), stream_handle(stream)))


def csa2_compress_workspace_size(B, T, H, d, Di) -> int:
    return lib().csa2_compress_workspace_size(B, T, H, d, Di)


def csa2_compress_pack(hidden, W, gamma, eps, rope_base, W_idx, first_entry, dims: Dims, cache: Cache,
                       ws, stream=None):
    B, T, H = hidden.shape
    _check(lib().csa2_compress_pack(ptr(hidden), B, T, H, ptr(W), ptr(gamma), eps, rope_base, ptr(W_idx),
                                    ptr(first_entry), C.byref(dims), C.byref(cache), ptr(ws),
                                    ws.numel() * ws.element_size() if ws is not None else 0,
                                    stream_handle(stream)))


def csa2_compress_layers_workspace_size(B, T, H, L, d, Di) -> int:
    return lib().csa2_compress_layers_workspace_size(B, T, H, L, d, Di)


def csa2_compress_layers(hidden, W_all, Di, gamma_all, eps, rope_base, first_entry, dims: Dims, caches, ws,
                         stream=None):
    """caches: a sequence of Cache (one per layer); W_all [L][d + Di][4H]; gamma_all [L][d]."""
    B, T, H = hidden.shape
    L = W_all.shape[0]
    arr = (Cache * L)(*caches)
    _check(lib().csa2_compress_layers(ptr(hidden), B, T, H, L, ptr(W_all), Di, ptr(gamma_all), eps, rope_base,
                                      ptr(first_entry), C.byref(dims), arr, ptr(ws),
                                      ws.numel() * ws.element_size() if ws is not None else 0,
                                      stream_handle(stream)))


def csa2_swa_replay_workspace_size(B, n_tok, H, d) -> int:
    return lib().csa2_swa_replay_workspace_size(B, n_tok, H, d)


def csa2_swa_replay(hidden, W_swa, gamma, eps, rope_base, tok_pos0, dims: Dims, window: Window, ws, stream=None):
    """hidden [B][n_tok][H] bf16 of the replayed tokens; W_swa [d][H] bf16; tok_pos0 int32 [B]."""
    B, n_tok, H = hidden.shape
    _check(lib().csa2_swa_replay(ptr(hidden), B, n_tok, H, ptr(W_swa), ptr(gamma), eps, rope_base, ptr(tok_pos0),
                                 C.byref(dims), C.byref(window), ptr(ws),
                                 ws.numel() * ws.element_size() if ws is not None else 0, stream_handle(stream)))


def csa2_index_scores(dims: Dims, cache: Cache, idx_q, w, q_pos, scores, blockmax=None, stream=None):
    _check(lib().csa2_index_scores(C.byref(dims), C.byref(cache), ptr(idx_q), ptr(w), ptr(q_pos),
                                   ptr(scores), scores.shape[-1], ptr(blockmax),
                                   blockmax.shape[-1] if blockmax is not None else 0, stream_handle(stream)))


def csa2_topk_workspace_size(rows, stride, k) -> int:
    return lib().csa2_topk_workspace_size(rows, stride, k)


def csa2_topk_f32(scores, n_valid, k, out_idx, out_cnt, ws=None, stream=None):
    rows, stride = scores.shape
    _check(lib().csa2_topk_f32(ptr(scores), rows, stride, ptr(n_valid), k, ptr(out_idx), ptr(out_cnt),
                               ptr(ws), ws.numel() * ws.element_size() if ws is not None else 0,
                               stream_handle(stream)))


def csa2_block_pool_f32(scores, n_valid, block, n_pool_blocks, out_pool, out_pool_cnt, out_blockmax=None,
                        ws=None, stream=None):
    rows, stride = scores.shape
    _check(lib().csa2_block_pool_f32(ptr(scores), rows, stride, ptr(n_valid), block, n_pool_blocks,
                                     ptr(out_pool), ptr(out_pool_cnt), ptr(out_blockmax), ptr(ws),
                                     ws.numel() * ws.element_size() if ws is not None else 0,
                                     stream_handle(stream)))


def csa2_index_topk_workspace_size(dims: Dims, max_entries: int) -> int:
    return lib().csa2_index_topk_workspace_size(C.byref(dims), max_entries)


def csa2_index_topk(dims: Dims, cache: Cache, idx_q, w, q_pos, out_idx, out_cnt, max_entries, ws,
                    pool=None, pool_cnt=None, out_pool=None, out_pool_cnt=None, stream=None):
    _check(lib().csa2_index_topk(C.byref(dims), C.byref(cache), ptr(idx_q), ptr(w), ptr(q_pos), ptr(pool),
                                 ptr(pool_cnt), ptr(out_idx), ptr(out_cnt), ptr(out_pool), ptr(out_pool_cnt),
                                 max_entries, ptr(ws), ws.numel() * ws.element_size(), stream_handle(stream)))


def csa2_index_topk_noalloc_capacity() -> int:
    return lib().csa2_index_topk_noalloc_capacity()


def csa2_index_topk_noalloc(dims: Dims, cache: Cache, idx_q, w, q_pos, out_idx, out_cnt, max_entries,
                            pool=None, pool_cnt=None, out_pool=None, out_pool_cnt=None, stream=None):
    """csa2_index_topk for callers that cannot allocate: scratch is the library's fixed device array."""
    _check(lib().csa2_index_topk_noalloc(C.byref(dims), C.byref(cache), ptr(idx_q), ptr(w), ptr(q_pos), ptr(pool),
                                         ptr(pool_cnt), ptr(out_idx), ptr(out_cnt), ptr(out_pool),
                                         ptr(out_pool_cnt), max_entries, stream_handle(stream)))


def csa2_sparse_attn(dims: Dims, cache: Cache, window: Window, Q, q_pos, idx, cnt, softmax_scale, O,
                     lse=None, stream=None):
    _check(lib().csa2_sparse_attn(C.byref(dims), C.byref(cache), C.byref(window), ptr(Q), ptr(q_pos),
                                  ptr(idx), ptr(cnt), softmax_scale, ptr(O), ptr(lse), stream_handle(stream)))


def csa2_layer_workspace_size(args: LayerArgs) -> int:
    return lib().csa2_layer_workspace_size(C.byref(args))


def csa2_layer(args: LayerArgs, ws, stream=None):
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().csa2_layer(C.byref(args), ptr(ws), nbytes, stream_handle(stream)))
