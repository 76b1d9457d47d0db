"""Thin ctypes binding over libb300attn.so (argument marshalling only).

Every function takes torch tensors that already live on the GPU, passes their
device pointers, sizes and the current CUDA stream to the C ABI declared in
include/b300attn.h, and raises B300AttnError on a non-OK status.  No step of
the computation runs here; torch only provides device memory and streams.
Importing this module fails loudly if the library has not been built.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
RELEASE_LIB_PATH = os.path.join(_HERE, "libb300attn.so")
# B300ATTN_DEBUG=1 selects the debug build (device-side checks reported by
# attn_device_status; built by `python -m ...build --debug`)
DEBUG_LIB_PATH = os.path.join(_HERE, "libb300attn_debug.so")
LIB_PATH = DEBUG_LIB_PATH if os.environ.get("B300ATTN_DEBUG") == "1" else RELEASE_LIB_PATH

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
BF16, F32 = 0, 1

# name -> (restype, argtypes) for every entry point of include/b300attn.h
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I]),
    "attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P,
                             _I]),
    "attn_fwd_paged": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                            _F, _P, _I]),
    "attn_bwd_workspace_size": (_SZ, [_I, _I, _I]),
    "attn_fp8_padded_len": (_I, [_I]),
    "attn_fp8_workspace_size": (_SZ, [_I, _I, _I]),
    "attn_fp8_quantize": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ,
                               _P]),
    "attn_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P,
                          _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _I,
                      _F, _P, _I]),
    "attn_decode_chunk": (_I, [_I, _I]),
    "attn_decode_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "attn_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ,
                                 _P, _I]),
    "attn_decode_splitkv_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I,
                                         _P, _I]),
    "attn_decode_splitkv_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                       _F, _I, _P, _SZ, _P, _I]),
    "attn_decode_partials": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "lse_tree_combine": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I]),
    "attn_device_status": (_I, [_P]),
    "attn_selftest_bounded_wait": (_I, [ctypes.c_ulonglong, _P]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_version": (_I, []),
}


class B300AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"b300attn status {status}: {message}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with "
            "`python -m exact_transformer_attention_flashattention_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int) -> None:
    if rc != OK:
        raise B300AttnError(rc, _lib.attn_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _odtype(dtype) -> int:
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float32:
        return F32
    raise ValueError(f"output dtype must be bfloat16 or float32, got {dtype}")


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def attn_fwd(q, k, v, causal: bool = False, window: int = -1, scale: float | None = None,
             out=None, lse=None, out_dtype=torch.bfloat16, stream=None):
    """Prefill attention.  q [B,N,Hq,d], k/v [B,N,Hkv,d] bf16 -> (O [B,N,Hq,d], LSE [B,Hq,N])."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 4)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    _check(_lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d,
                         int(bool(causal)), int(window), float(scale), _stream(stream),
                         _odtype(out.dtype)))
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, window: int = -1,
                    scale: float | None = None, out=None, lse=None, out_dtype=torch.bfloat16,
                    stream=None):
    """Prefill over sequences packed back to back.  q [T,Hq,d], k/v [T,Hkv,d] bf16,
    cu_seqlens int32 [S+1] on the device -> (O [T,Hq,d], LSE [Hq,T])."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((T, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    S = cu_seqlens.numel() - 1
    _check(_lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
                                S, T, int(max_seqlen), Hq, Hkv, d, int(bool(causal)), int(window),
                                float(scale), _stream(stream), _odtype(out.dtype)))
    return out, lse


def attn_fwd_paged(q, k_pages, v_pages, block_table, causal: bool = False, window: int = -1,
                   scale: float | None = None, out=None, lse=None, out_dtype=torch.bfloat16,
                   stream=None):
    """Prefill with K/V in a page pool.  q [B,N,Hq,d] bf16; pages [P, page_size, Hkv, d]
    bf16; block_table int32 [B, pages_per_seq] -> (O [B,N,Hq,d], LSE [B,Hq,N])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    B, N, Hq, d = q.shape
    P, page_size, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if k_pages.shape != (P, page_size, Hkv, d) or v_pages.shape != k_pages.shape:
        raise ValueError("page pool shapes do not match q")
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per sequence")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    _check(_lib.attn_fwd_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                               _ptr(out), _ptr(lse), B, Hq, Hkv, N, d, page_size, P,
                               block_table.shape[1], int(bool(causal)), int(window), float(scale),
                               _stream(stream), _odtype(out.dtype)))
    return out, lse


def attn_bwd_workspace_size(B: int, Hq: int, N: int) -> int:
    return int(_lib.attn_bwd_workspace_size(B, Hq, N))


def attn_bwd(q, k, v, o, lse, dO, causal: bool = False, window: int = -1,
             scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of attn_fwd: q, dO [B,N,Hq,d], k/v [B,N,Hkv,d] bf16, o (bf16 or
    f32) and lse [B,Hq,N] from the forward -> (dQ, dK, dV) bf16."""
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _need(t, name, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape or dO.shape != q.shape:
        raise ValueError("shapes of k, v or dO do not match q")
    if o.shape != q.shape or not o.is_contiguous():
        raise ValueError("o must be a contiguous tensor shaped like q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_bwd_workspace_size(B, Hq, N)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                         _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, Hq, Hkv, N, d,
                         int(bool(causal)), int(window), float(scale), _stream(stream),
                         _odtype(o.dtype)))
    return dq, dk, dv


def attn_fp8_padded_len(N: int) -> int:
    return int(_lib.attn_fp8_padded_len(N))


def attn_fp8_workspace_size(B: int, Hkv: int, N: int) -> int:
    return int(_lib.attn_fp8_workspace_size(B, Hkv, N))


def attn_fp8_quantize(q, k, v, out=None, workspace=None, stream=None):
    """bf16 q [B,N,Hq,d], k/v [B,N,Hkv,d] -> dict of e4m3 codes (uint8 tensors)
    and int32 exponents: q8 [B,N,Hq,d], k8 [B,N,Hkv,d], v8t [B,Hkv,d,Np],
    q_exp [B,Hq,nt], k_exp [B,Hkv,nt], v_exp [B,Hkv] (nt = ceil(N/128)).
    ``out`` may hold preallocated tensors under the same names."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 4)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError(f"k/v shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    nt, Np = (N + 127) // 128, attn_fp8_padded_len(N)
    dev = q.device
    shapes = {"q8": ((B, N, Hq, d), torch.uint8), "k8": ((B, N, Hkv, d), torch.uint8),
              "v8t": ((B, Hkv, d, Np), torch.uint8), "q_exp": ((B, Hq, nt), torch.int32),
              "k_exp": ((B, Hkv, nt), torch.int32), "v_exp": ((B, Hkv), torch.int32)}
    out = dict(out or {})
    for name, (shape, dt) in shapes.items():
        if name not in out:
            out[name] = torch.empty(shape, dtype=dt, device=dev)
        t = out[name]
        if tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor of shape {shape}")
    need = attn_fp8_workspace_size(B, Hkv, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(_lib.attn_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), _ptr(out["q8"]), _ptr(out["k8"]),
                                  _ptr(out["v8t"]), _ptr(out["q_exp"]), _ptr(out["k_exp"]),
                                  _ptr(out["v_exp"]), B, Hq, Hkv, N, d, _ptr(workspace),
                                  workspace.numel(), _stream(stream)))
    return out


def attn_fwd_fp8(qz, causal: bool = False, window: int = -1, scale: float | None = None,
                 out=None, lse=None, out_dtype=torch.bfloat16, stream=None):
    """Prefill attention on the e4m3 operands of ``attn_fp8_quantize`` (the dict
    it returns) -> (O [B,N,Hq,d], LSE [B,Hq,N])."""
    q8, k8, v8t = qz["q8"], qz["k8"], qz["v8t"]
    for name, t, nd in (("q8", q8, 4), ("k8", k8, 4), ("v8t", v8t, 4)):
        _need(t, name, torch.uint8, nd)
    for name in ("q_exp", "k_exp", "v_exp"):
        _need(qz[name], name, torch.int32, 3 if name != "v_exp" else 2)
    B, N, Hq, d = q8.shape
    Hkv = k8.shape[2]
    if k8.shape != (B, N, Hkv, d) or v8t.shape != (B, Hkv, d, attn_fp8_padded_len(N)):
        raise ValueError("k8 / v8t shapes do not match q8")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, Hq, d), dtype=out_dtype, device=q8.device)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q8.device)
    _check(_lib.attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(qz["q_exp"]), _ptr(qz["k_exp"]),
                             _ptr(qz["v_exp"]), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d,
                             int(bool(causal)), int(window), float(scale), _stream(stream),
                             _odtype(out.dtype)))
    return out, lse


def attn_decode_chunk(max_kv_len: int, num_splits: int) -> int:
    c = _lib.attn_decode_chunk(max_kv_len, num_splits)
    _check(min(c, 0))
    return c


def attn_decode_workspace_size(B: int, Hq: int, num_splits: int, d: int) -> int:
    return int(_lib.attn_decode_workspace_size(B, Hq, num_splits, d))


def attn_decode_splitkv(q, k_cache, v_cache, kv_len, num_splits: int, scale: float | None = None,
                        out=None, lse=None, workspace=None, out_dtype=torch.bfloat16,
                        stream=None):
    """Split-KV decode.  q [B,Hq,d], caches [B,Lmax,Hkv,d] bf16, kv_len int32 [B]
    -> (O [B,Hq,d], LSE [B,Hq]).  ``workspace`` (uint8, optional) receives the
    split partials."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(kv_len, "kv_len", torch.int32, 1)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Lmax, Hkv, d) or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes do not match q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, num_splits, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
                                    _ptr(out), _ptr(lse), B, Hq, Hkv, Lmax, d, float(scale),
                                    int(num_splits), _ptr(workspace), workspace.numel(),
                                    _stream(stream), _odtype(out.dtype)))
    return out, lse


def attn_decode_splitkv_noalloc(q, k_cache, v_cache, kv_len, num_splits: int,
                                scale: float | None = None, out=None, lse=None,
                                out_dtype=torch.bfloat16, stream=None):
    """Split-KV decode whose split partials live in the library's built-in
    scratch (no workspace argument; the library allocates nothing).  For
    callers that must not allocate device memory when they run decode.  Calls
    share the scratch: do not let two of them overlap on the GPU."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(kv_len, "kv_len", torch.int32, 1)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Lmax, Hkv, d) or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes do not match q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(_lib.attn_decode_splitkv_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
                                            _ptr(out), _ptr(lse), B, Hq, Hkv, Lmax, d,
                                            float(scale), int(num_splits), _stream(stream),
                                            _odtype(out.dtype)))
    return out, lse


def attn_decode_splitkv_paged(q, k_pages, v_pages, block_table, kv_len, num_splits: int,
                              scale: float | None = None, out=None, lse=None, workspace=None,
                              out_dtype=torch.bfloat16, stream=None):
    """Split-KV decode over a paged cache.  q [B,Hq,d]; pages [P, page_size, Hkv, d]
    bf16; block_table int32 [B, pages_per_seq]; kv_len int32 [B] -> (O, LSE)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(kv_len, "kv_len", torch.int32, 1)
    B, Hq, d = q.shape
    P, page_size, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if k_pages.shape != (P, page_size, Hkv, d) or v_pages.shape != k_pages.shape:
        raise ValueError("page pool shapes do not match q")
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per sequence")
    pps = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, num_splits, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_decode_splitkv_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages),
                                          _ptr(block_table), _ptr(kv_len), _ptr(out), _ptr(lse),
                                          B, Hq, Hkv, page_size, P, pps, d, float(scale),
                                          int(num_splits), _ptr(workspace), workspace.numel(),
                                          _stream(stream), _odtype(out.dtype)))
    return out, lse


def attn_decode_partials(q, k_cache, v_cache, kv_len, num_splits: int,
                         scale: float | None = None, workspace=None, stream=None):
    """Split partials only (no merge).  Returns the workspace; read it with
    ``split_partials_view``."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(kv_len, "kv_len", torch.int32, 1)
    B, Hq, d = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Lmax, Hkv, d) or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes do not match q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_size(B, Hq, num_splits, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(_lib.attn_decode_partials(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), B, Hq,
                                     Hkv, Lmax, d, float(scale), int(num_splits), _ptr(workspace),
                                     workspace.numel(), _stream(stream)))
    return workspace


def split_partials_view(workspace, B: int, Hq: int, num_splits: int, d: int):
    """(m, l, o) views of a decode workspace: [B*Hq, S], [B*Hq, S], [B*Hq, S, d] f32."""
    rows = B * Hq * num_splits
    a = (rows * 4 + 255) // 256 * 256
    f = workspace.view(torch.uint8)
    m = f[:rows * 4].view(torch.float32).view(B * Hq, num_splits)
    l = f[a:a + rows * 4].view(torch.float32).view(B * Hq, num_splits)
    o = f[2 * a:2 * a + rows * d * 4].view(torch.float32).view(B * Hq, num_splits, d)
    return m, l, o


def lse_tree_combine(part_m, part_l, part_o, out=None, lse=None, out_dtype=torch.float32,
                     stream=None):
    """Merge split partials: m, l [R,S], o [R,S,d] f32 -> (O [R,d], LSE [R])."""
    _need(part_m, "part_m", torch.float32, 2)
    _need(part_l, "part_l", torch.float32, 2)
    _need(part_o, "part_o", torch.float32, 3)
    R, S = part_m.shape
    d = part_o.shape[2]
    if out is None:
        out = torch.empty((R, d), dtype=out_dtype, device=part_m.device)
    if lse is None:
        lse = torch.empty((R,), dtype=torch.float32, device=part_m.device)
    _check(_lib.lse_tree_combine(_ptr(part_m), _ptr(part_l), _ptr(part_o), _ptr(out), _ptr(lse),
                                 R, S, d, _stream(stream), _odtype(out.dtype)))
    return out, lse


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device status."""
    return int(_lib.attn_device_status(_stream(stream)))


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch the library's failure-path self-test: a wait that nothing ends
    gives up after ``limit_ns``; the next ``device_status`` reports it."""
    _check(_lib.attn_selftest_bounded_wait(int(limit_ns), _stream(stream)))


def last_error() -> str:
    return _lib.attn_last_error().decode()
