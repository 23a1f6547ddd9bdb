"""ctypes binding of libpkv.so (include/pkv.h), one Python function per C entry point.

Argument marshalling only: torch tensors are passed as raw device pointers on
the current CUDA stream, host arrays as raw host pointers. Before a device
pointer is handed to a kernel the binding checks that the tensor lives on a
CUDA device, is contiguous, and is large enough for the sizes passed -- the C
ABI cannot see buffer sizes, and a wrong pointer must never reach a kernel.
A nonzero status becomes a ``PkvError``. There is no fallback: if the library
is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID = -1
PKV_ERR_OOM = -2
PKV_ERR_NOT_FOUND = -3
PKV_ERR_EXISTS = -4
PKV_ERR_UNSUPPORTED = -5
PKV_ERR_CUDA = -6
PKV_ERR_DEVICE_TIMEOUT = -7
PKV_ERR_TOO_LARGE = -8
PKV_STATIC_WS_BYTES = 8 << 20

PKV_DEVERR_BLOCK_ID = 1
PKV_DEVERR_SLOT = 2
PKV_DEVERR_CTX_LEN = 4
PKV_DEVERR_OFFSET = 8
PKV_DEVERR_TIMEOUT = 16

PKV_DTYPE_BF16 = 0
PKV_DTYPE_INT8 = 1

_NAMES = {PKV_ERR_INVALID: "PKV_ERR_INVALID", PKV_ERR_OOM: "PKV_ERR_OOM",
          PKV_ERR_NOT_FOUND: "PKV_ERR_NOT_FOUND", PKV_ERR_EXISTS: "PKV_ERR_EXISTS",
          PKV_ERR_UNSUPPORTED: "PKV_ERR_UNSUPPORTED", PKV_ERR_CUDA: "PKV_ERR_CUDA",
          PKV_ERR_DEVICE_TIMEOUT: "PKV_ERR_DEVICE_TIMEOUT", PKV_ERR_TOO_LARGE: "PKV_ERR_TOO_LARGE"}

EXPORTED = (
    "pkv_allocator_create", "pkv_allocator_destroy", "pkv_alloc", "pkv_append_block", "pkv_free",
    "pkv_attach_shared", "pkv_num_free", "pkv_request_table", "pkv_free_list",
    "pkv_build_block_tables", "pkv_append_kv", "pkv_quantize_full_blocks",
    "pkv_quantize_blocks_from", "pkv_decode_attention", "pkv_splitk_reduce",
    "pkv_splitk_ws_o_bytes", "pkv_splitk_ws_ml_bytes", "pkv_decode_ctas_per_sm",
    "pkv_decode_attention_static_ws", "pkv_set_programmatic_launch", "pkv_decode_step", "pkv_decode_layers",
    "pkv_fork", "pkv_cow_block", "pkv_block_refs", "pkv_copy_blocks", "pkv_copy_slots",
    "pkv_debug_skip_copy", "pkv_sync_status",
)


class PkvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {_NAMES.get(code, code)}")
        self.code = code


class CacheDesc(ctypes.Structure):
    """Mirror of ``pkv_cache_desc``."""
    _fields_ = [
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("scales", ctypes.c_void_p),
        ("k_tail", ctypes.c_void_p), ("v_tail", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("max_slots", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("err_word", ctypes.c_void_p),
    ]


_lib = None
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with paged_kv_cache_56_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "pkv_allocator_create": (_VP, [_I32, _I32, _I32P]),
            "pkv_allocator_destroy": (None, [_VP]),
            "pkv_alloc": (ctypes.c_int, [_VP, _I64, _I32, _I32P]),
            "pkv_append_block": (ctypes.c_int, [_VP, _I64, _I32P]),
            "pkv_free": (ctypes.c_int, [_VP, _I64]),
            "pkv_attach_shared": (ctypes.c_int, [_VP, _I64, _I32P, _I32]),
            "pkv_fork": (ctypes.c_int, [_VP, _I64, _I64]),
            "pkv_cow_block": (ctypes.c_int, [_VP, _I64, _I32, _I32P, _I32P]),
            "pkv_block_refs": (ctypes.c_int, [_VP, _I32]),
            "pkv_copy_blocks": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _I32, _VP]),
            "pkv_copy_slots": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _I32, _VP]),
            "pkv_sync_status": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _I32, _VP, _I32P]),
            "pkv_num_free": (ctypes.c_int, [_VP]),
            "pkv_request_table": (ctypes.c_int, [_VP, _I64, _I32P, _I32]),
            "pkv_free_list": (ctypes.c_int, [_VP, _I32P, _I32]),
            "pkv_build_block_tables": (ctypes.c_int, [_VP, _I64P, _I32, _I32, _I32P]),
            "pkv_append_kv": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _VP, _VP, _VP, _I32, _VP]),
            "pkv_quantize_full_blocks": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _I32, _VP]),
            "pkv_quantize_blocks_from": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _VP, _I32, _VP]),
            "pkv_decode_attention": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _I32, _VP, _VP, _I32,
                                                    ctypes.c_float, _I32, _I32, _VP, _VP, _VP, _VP, _VP]),
            "pkv_decode_ctas_per_sm": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _I32, _I32]),
            "pkv_set_programmatic_launch": (ctypes.c_int, [ctypes.c_int]),
            "pkv_debug_skip_copy": (ctypes.c_int, [_I32]),
            "pkv_decode_layers": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _I32, _VP, _I64, _VP, _VP, _I64, _VP,
                                                 _I64, _VP, _I32, _VP, _VP, _I32, ctypes.c_float, _I32, _I32, _VP,
                                                 _VP, _VP, _VP]),
            "pkv_decode_step": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _VP, _VP, _I32, _VP, _VP, _I32,
                                               ctypes.c_float, _I32, _I32, _VP, _VP, _VP, _VP, _VP]),
            "pkv_decode_attention_static_ws": (ctypes.c_int, [ctypes.POINTER(CacheDesc), _VP, _VP, _I32, _VP, _VP,
                                                              _I32, ctypes.c_float, _I32, _I32, _VP, _VP]),
            "pkv_splitk_reduce": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP]),
            "pkv_splitk_ws_o_bytes": (ctypes.c_size_t, [_I32, _I32, _I32, _I32]),
            "pkv_splitk_ws_ml_bytes": (ctypes.c_size_t, [_I32, _I32, _I32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(fn: str, rc: int) -> None:
    if rc != PKV_OK:
        raise PkvError(fn, rc)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype, min_numel: int = 0) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {min_numel}")
    return t.data_ptr()


def _opt_dev(t, name, dtype, min_numel=0) -> int | None:
    return None if t is None else _dev(t, name, dtype, min_numel)


def _host_i32(a, n=None) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))
    if n is not None and a.size < n:
        raise ValueError("host array too short")
    return a


# ---------------------------------------------------------------------------
# Host allocator
# ---------------------------------------------------------------------------

def pkv_allocator_create(num_blocks: int, block_size: int, initial_order=None):
    order = None
    if initial_order is not None:
        order = _host_i32(initial_order, num_blocks)
        if order.size != num_blocks:
            raise ValueError("initial_order must have num_blocks entries")
    h = lib().pkv_allocator_create(num_blocks, block_size,
                                   None if order is None else order.ctypes.data_as(_I32P))
    if not h:
        raise PkvError("pkv_allocator_create", PKV_ERR_INVALID)
    return ctypes.c_void_p(h)


def pkv_allocator_destroy(h) -> None:
    lib().pkv_allocator_destroy(h)


def pkv_alloc(h, req_id: int, n_blocks: int) -> list:
    out = np.empty(max(n_blocks, 1), dtype=np.int32)
    _check("pkv_alloc", lib().pkv_alloc(h, req_id, n_blocks, out.ctypes.data_as(_I32P)))
    return out[:n_blocks].tolist()


def pkv_append_block(h, req_id: int) -> int:
    out = ctypes.c_int32(-1)
    _check("pkv_append_block", lib().pkv_append_block(h, req_id, ctypes.byref(out)))
    return out.value


def pkv_free(h, req_id: int) -> None:
    _check("pkv_free", lib().pkv_free(h, req_id))


def pkv_fork(h, parent: int, child: int) -> None:
    _check("pkv_fork", lib().pkv_fork(h, parent, child))


def pkv_cow_block(h, req_id: int, index: int):
    """(old, new) block ids if a private copy replaced a shared block, else None."""
    src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
    _check("pkv_cow_block", lib().pkv_cow_block(h, req_id, index, ctypes.byref(src), ctypes.byref(dst)))
    return None if src.value < 0 else (src.value, dst.value)


def pkv_block_refs(h, block: int) -> int:
    rc = lib().pkv_block_refs(h, block)
    if rc < 0:
        raise PkvError("pkv_block_refs", rc)
    return rc


def pkv_attach_shared(h, req_id: int, ids) -> None:
    a = _host_i32(ids)
    _check("pkv_attach_shared", lib().pkv_attach_shared(h, req_id, a.ctypes.data_as(_I32P), a.size))


def pkv_num_free(h) -> int:
    return lib().pkv_num_free(h)


def pkv_request_table(h, req_id: int) -> list:
    n = lib().pkv_request_table(h, req_id, None, 0)
    if n < 0:
        raise PkvError("pkv_request_table", n)
    out = np.empty(max(n, 1), dtype=np.int32)
    lib().pkv_request_table(h, req_id, out.ctypes.data_as(_I32P), n)
    return out[:n].tolist()


def pkv_free_list(h) -> list:
    n = lib().pkv_free_list(h, None, 0)
    if n < 0:
        raise PkvError("pkv_free_list", n)
    out = np.empty(max(n, 1), dtype=np.int32)
    lib().pkv_free_list(h, out.ctypes.data_as(_I32P), n)
    return out[:n].tolist()


def pkv_build_block_tables(h, req_ids, max_blocks: int, out: np.ndarray | None = None) -> np.ndarray:
    """Returns (or fills) a host int32 array [B, max_blocks]."""
    ids = np.ascontiguousarray(np.asarray(req_ids, dtype=np.int64).reshape(-1))
    B = ids.size
    if out is None:
        out = np.empty((B, max_blocks), dtype=np.int32)
    if out.dtype != np.int32 or not out.flags.c_contiguous or out.size < B * max_blocks:
        raise ValueError("out must be a C-contiguous int32 array of B * max_blocks entries")
    _check("pkv_build_block_tables",
           lib().pkv_build_block_tables(h, ids.ctypes.data_as(_I64P), B, max_blocks, out.ctypes.data_as(_I32P)))
    return out


# ---------------------------------------------------------------------------
# Device entry points
# ---------------------------------------------------------------------------

def _desc_ptr(desc: CacheDesc):
    return ctypes.byref(desc)


def pkv_append_kv(desc: CacheDesc, k: torch.Tensor, v: torch.Tensor, block_ids, offsets, slots,
                  stream=None) -> None:
    T = k.shape[0] if k.dim() else 0
    row = desc.num_kv_heads * desc.head_dim
    kp = _dev(k, "k", torch.bfloat16, T * row)
    vp = _dev(v, "v", torch.bfloat16, T * row)
    int8 = desc.dtype == PKV_DTYPE_INT8
    bp = _opt_dev(block_ids, "block_ids", torch.int32, 0 if int8 else T)
    sp = _opt_dev(slots, "slots", torch.int32, T if int8 else 0)
    op = _dev(offsets, "offsets", torch.int32, T)
    _check("pkv_append_kv", lib().pkv_append_kv(_desc_ptr(desc), kp, vp, bp, op, sp, T, _stream(stream)))


def pkv_quantize_full_blocks(desc: CacheDesc, block_ids: torch.Tensor, slots: torch.Tensor,
                             stream=None) -> None:
    M = block_ids.numel()
    bp = _dev(block_ids, "block_ids", torch.int32, M)
    sp = _dev(slots, "slots", torch.int32, M)
    _check("pkv_quantize_full_blocks",
           lib().pkv_quantize_full_blocks(_desc_ptr(desc), bp, sp, M, _stream(stream)))


def pkv_copy_blocks(desc: CacheDesc, src_ids: torch.Tensor, dst_ids: torch.Tensor, stream=None) -> None:
    n = src_ids.numel()
    sp = _dev(src_ids, "src_ids", torch.int32, n)
    dp = _dev(dst_ids, "dst_ids", torch.int32, n)
    _check("pkv_copy_blocks", lib().pkv_copy_blocks(_desc_ptr(desc), sp, dp, n, _stream(stream)))


def pkv_copy_slots(desc: CacheDesc, src_slots: torch.Tensor, dst_slots: torch.Tensor, stream=None) -> None:
    n = src_slots.numel()
    sp = _dev(src_slots, "src_slots", torch.int32, n)
    dp = _dev(dst_slots, "dst_slots", torch.int32, n)
    _check("pkv_copy_slots", lib().pkv_copy_slots(_desc_ptr(desc), sp, dp, n, _stream(stream)))


def pkv_quantize_blocks_from(desc: CacheDesc, k_src: torch.Tensor, v_src: torch.Tensor,
                             block_ids: torch.Tensor, stream=None) -> None:
    M = block_ids.numel()
    need = M * desc.block_size * desc.num_kv_heads * desc.head_dim
    kp = _dev(k_src, "k_src", torch.bfloat16, need)
    vp = _dev(v_src, "v_src", torch.bfloat16, need)
    bp = _dev(block_ids, "block_ids", torch.int32, M)
    _check("pkv_quantize_blocks_from",
           lib().pkv_quantize_blocks_from(_desc_ptr(desc), kp, vp, bp, M, _stream(stream)))


def pkv_debug_skip_copy(tile: int) -> None:
    """Test hook: later decode launches leave one tile's copies unissued so that a
    bounded wait runs out (PKV_DEVERR_TIMEOUT); -1 turns it off."""
    _check("pkv_debug_skip_copy", lib().pkv_debug_skip_copy(tile))


def pkv_set_programmatic_launch(enable: bool) -> None:
    _check("pkv_set_programmatic_launch", lib().pkv_set_programmatic_launch(1 if enable else 0))


def pkv_splitk_ws_o_bytes(B: int, Hq: int, head_dim: int, max_splits: int) -> int:
    return lib().pkv_splitk_ws_o_bytes(B, Hq, head_dim, max_splits)


def pkv_splitk_ws_ml_bytes(B: int, Hq: int, max_splits: int) -> int:
    return lib().pkv_splitk_ws_ml_bytes(B, Hq, max_splits)


def pkv_decode_ctas_per_sm(desc: CacheDesc, split_tokens: int, max_blocks: int) -> int:
    n = lib().pkv_decode_ctas_per_sm(_desc_ptr(desc), split_tokens, max_blocks)
    if n < 0:
        raise PkvError("pkv_decode_ctas_per_sm", n)
    return n


def pkv_decode_attention(desc: CacheDesc, q: torch.Tensor, block_tables: torch.Tensor,
                         ctx_lens: torch.Tensor, slots, sm_scale: float, out: torch.Tensor,
                         split_tokens: int = 0, max_splits: int = 0, ws_o=None, ws_ml=None,
                         ws_count=None, stream=None) -> None:
    B = ctx_lens.numel()
    max_blocks = block_tables.shape[-1] if block_tables.dim() == 2 else 0
    hq, d = desc.num_q_heads, desc.head_dim
    qp = _dev(q, "q", torch.bfloat16, B * hq * d)
    outp = _dev(out, "out", torch.bfloat16, B * hq * d)
    tp = _dev(block_tables, "block_tables", torch.int32, B * max_blocks)
    cp = _dev(ctx_lens, "ctx_lens", torch.int32, B)
    sp = _opt_dev(slots, "slots", torch.int32, B)
    wo = wml = wc = None
    if split_tokens > 0:
        wo = _dev(ws_o, "ws_o", torch.float32, B * hq * max_splits * d)
        wml = _dev(ws_ml, "ws_ml", torch.float32, B * hq * max_splits * 2)
        wc = _opt_dev(ws_count, "ws_count", torch.int32, B * desc.num_kv_heads)
    _check("pkv_decode_attention",
           lib().pkv_decode_attention(_desc_ptr(desc), qp, tp, max_blocks, cp, sp, B, float(sm_scale),
                                      split_tokens, max_splits, wo, wml, wc, outp, _stream(stream)))


def pkv_decode_step(desc: CacheDesc, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    block_tables: torch.Tensor, ctx_lens: torch.Tensor, slots, sm_scale: float, out: torch.Tensor,
                    split_tokens: int = 0, max_splits: int = 0, ws_o=None, ws_ml=None, ws_count=None,
                    stream=None) -> None:
    B = ctx_lens.numel()
    max_blocks = block_tables.shape[-1] if block_tables.dim() == 2 else 0
    hq, hkv, d = desc.num_q_heads, desc.num_kv_heads, desc.head_dim
    qp = _dev(q, "q", torch.bfloat16, B * hq * d)
    kp = _dev(k_new, "k_new", torch.bfloat16, B * hkv * d)
    vp = _dev(v_new, "v_new", torch.bfloat16, B * hkv * d)
    outp = _dev(out, "out", torch.bfloat16, B * hq * d)
    tp = _dev(block_tables, "block_tables", torch.int32, B * max_blocks)
    cp = _dev(ctx_lens, "ctx_lens", torch.int32, B)
    sp = _opt_dev(slots, "slots", torch.int32, B)
    wo = wml = wc = None
    if split_tokens > 0:
        wo = _dev(ws_o, "ws_o", torch.float32, B * hq * max_splits * d)
        wml = _dev(ws_ml, "ws_ml", torch.float32, B * hq * max_splits * 2)
        wc = _opt_dev(ws_count, "ws_count", torch.int32, B * hkv)
    _check("pkv_decode_step",
           lib().pkv_decode_step(_desc_ptr(desc), qp, kp, vp, tp, max_blocks, cp, sp, B, float(sm_scale),
                                 split_tokens, max_splits, wo, wml, wc, outp, _stream(stream)))


def _layered(t: torch.Tensor, name: str, L: int, inner) -> int:
    """Device pointer of a [>=L, *inner] bf16 tensor whose per-layer slices are
    contiguous (the layer stride may exceed the slice, e.g. a batch slice of a
    larger buffer); checks that every slice lies inside the storage."""
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda" or t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be a bf16 CUDA tensor")
    if t.dim() != 1 + len(inner) or t.shape[0] < L or tuple(t.shape[1:]) != tuple(inner):
        raise ValueError(f"{name} must be [{L}, {', '.join(map(str, inner))}], got {tuple(t.shape)}")
    n = 1
    for x in inner:
        n *= x
    if not t[0].is_contiguous() or t.stride(0) < n:
        raise ValueError(f"{name}: each layer's slice must be contiguous")
    span = (L - 1) * t.stride(0) + n
    avail = t.untyped_storage().nbytes() // 2 - t.storage_offset()
    if span > avail:
        raise ValueError(f"{name} does not hold {L} layers")
    return t.data_ptr()


def desc_array(descs) -> ctypes.Array:
    """A contiguous C array of descriptors (one per layer) for pkv_decode_layers."""
    arr = (CacheDesc * len(descs))()
    for i, d in enumerate(descs):
        ctypes.memmove(ctypes.byref(arr, i * ctypes.sizeof(CacheDesc)), ctypes.byref(d), ctypes.sizeof(CacheDesc))
    return arr


def pkv_decode_layers(descs: ctypes.Array, q: torch.Tensor, k_new, v_new, block_tables: torch.Tensor,
                      ctx_lens: torch.Tensor, slots, sm_scale: float, out: torch.Tensor, split_tokens: int = 0,
                      max_splits: int = 0, ws_o=None, ws_ml=None, ws_count=None, stream=None) -> None:
    """Decode step over all layers in one call. q, out: [L, B, Hq, d]; k_new,
    v_new: [L, B, Hkv, d] or None (attention only); descs from desc_array()."""
    L = len(descs)
    B = ctx_lens.numel()
    d0 = descs[0]
    hq, hkv, d = d0.num_q_heads, d0.num_kv_heads, d0.head_dim
    qp = _layered(q, "q", L, (B, hq, d))
    outp = _layered(out, "out", L, (B, hq, d))
    kp = vp = None
    kv_stride = 0
    if k_new is not None:
        if v_new is None or v_new.stride(0) != k_new.stride(0):
            raise ValueError("k_new and v_new must be given together, with the same layer stride")
        kp = _layered(k_new, "k_new", L, (B, hkv, d))
        vp = _layered(v_new, "v_new", L, (B, hkv, d))
        kv_stride = k_new.stride(0) * 2
    max_blocks = block_tables.shape[-1] if block_tables.dim() == 2 else 0
    tp = _dev(block_tables, "block_tables", torch.int32, B * max_blocks)
    cp = _dev(ctx_lens, "ctx_lens", torch.int32, B)
    sp = _opt_dev(slots, "slots", torch.int32, B)
    wo = wml = wc = None
    if split_tokens > 0:
        wo = _dev(ws_o, "ws_o", torch.float32, B * hq * max_splits * d)
        wml = _dev(ws_ml, "ws_ml", torch.float32, B * hq * max_splits * 2)
        wc = _opt_dev(ws_count, "ws_count", torch.int32, B * hkv)
    _check("pkv_decode_layers",
           lib().pkv_decode_layers(descs, L, qp, q.stride(0) * 2, kp, vp, kv_stride, outp, out.stride(0) * 2, tp,
                                   max_blocks, cp, sp, B, float(sm_scale), split_tokens, max_splits, wo, wml, wc,
                                   _stream(stream)))


def pkv_splitk_reduce(ws_o: torch.Tensor, ws_ml: torch.Tensor, ctx_lens: torch.Tensor, num_q_heads: int,
                      head_dim: int, split_tokens: int, max_splits: int, out: torch.Tensor,
                      stream=None) -> None:
    B = ctx_lens.numel()
    wo = _dev(ws_o, "ws_o", torch.float32, B * num_q_heads * max_splits * head_dim)
    wml = _dev(ws_ml, "ws_ml", torch.float32, B * num_q_heads * max_splits * 2)
    cp = _dev(ctx_lens, "ctx_lens", torch.int32, B)
    op = _dev(out, "out", torch.bfloat16, B * num_q_heads * head_dim)
    _check("pkv_splitk_reduce",
           lib().pkv_splitk_reduce(wo, wml, cp, B, num_q_heads, head_dim, split_tokens, max_splits, op,
                                   _stream(stream)))


def pkv_decode_attention_static_ws(desc: CacheDesc, q: torch.Tensor, block_tables: torch.Tensor,
                                   ctx_lens: torch.Tensor, slots, sm_scale: float, out: torch.Tensor,
                                   split_tokens: int, max_splits: int, stream=None) -> None:
    """pkv_decode_attention with the split-K scratch in the library's fixed
    array: allocates nothing (see include/pkv.h for the size limit and the
    rule that overlapping calls race)."""
    B = ctx_lens.numel()
    max_blocks = block_tables.shape[-1] if block_tables.dim() == 2 else 0
    hq, d = desc.num_q_heads, desc.head_dim
    qp = _dev(q, "q", torch.bfloat16, B * hq * d)
    outp = _dev(out, "out", torch.bfloat16, B * hq * d)
    tp = _dev(block_tables, "block_tables", torch.int32, B * max_blocks)
    cp = _dev(ctx_lens, "ctx_lens", torch.int32, B)
    sp = _opt_dev(slots, "slots", torch.int32, B)
    _check("pkv_decode_attention_static_ws",
           lib().pkv_decode_attention_static_ws(_desc_ptr(desc), qp, tp, max_blocks, cp, sp, B, float(sm_scale),
                                                split_tokens, max_splits, outp, _stream(stream)))


def pkv_sync_status(descs, stream=None, raise_on_error: bool = True) -> int:
    """Waits for ``stream``, reads and clears the error words of ``descs`` (one
    CacheDesc or a sequence of them) and returns the OR of their PKV_DEVERR_*
    bits. With raise_on_error, a nonzero status (PKV_ERR_DEVICE_TIMEOUT for an
    expired bounded wait, PKV_ERR_INVALID for an out-of-range value in device
    memory) raises PkvError after the words have been cleared."""
    if isinstance(descs, CacheDesc):
        descs = [descs]
    arr = descs if isinstance(descs, ctypes.Array) else desc_array(list(descs))
    bits = ctypes.c_int32(0)
    rc = lib().pkv_sync_status(arr, len(arr), _stream(stream), ctypes.byref(bits))
    if raise_on_error:
        _check("pkv_sync_status", rc)
    elif rc not in (PKV_OK, PKV_ERR_DEVICE_TIMEOUT, PKV_ERR_INVALID):
        _check("pkv_sync_status", rc)
    return bits.value
