"""GB300 (sm_103a) quantize-and-scatter library for a paged MLA KV cache.

Python binding of the C ABI in include/kvq.h. Every function here only
marshals torch tensors into pointers, sizes and the current CUDA stream and
calls the same-named entry point of libkvq.so; all work runs in the CUDA
kernels. There is no fallback: if the library is not built, importing the
functions works but every call raises. Tensors are CUDA tensors, or pinned
CPU tensors that the device addresses at the same pointer (the kernels then
read and write host memory over the host-device link, with no copies).

  mxfp4_mla_store            quantize bf16 latent rows to 272-byte MXFP4 rows
  mxfp4_mla_rmsnorm_store    RMSNorm (bf16 weight, eps) then the MXFP4 store, one pass
  rope_quant_insert_mxfp8    GPT-J RoPE then the 528-byte MXFP8 record
  rope_quant_insert_nvfp4    GPT-J RoPE then the 288-byte NVFP4 record
  mxfp4_mla_gather_dequant   gather packed rows back to bf16
  mxfp4_mla_sparse_attention sparse MLA decode attention on the packed cache
"""
import contextlib
import ctypes
import os

import torch

__all__ = ["mxfp4_mla_store", "mxfp4_mla_rmsnorm_store", "rope_quant_insert_mxfp8",
           "rope_quant_insert_nvfp4", "rope_quant_insert_v4", "rope_plain_insert",
           "save_ring_rows", "fused_save_compress_norm",
           "mxfp4_mla_gather_dequant", "mxfp4_mla_sparse_attention", "attention_workspace_size",
           "attention_prefers_split", "mxfp4_mla_sparse_attention_ragged",
           "row_bytes",
           "cache_view", "KvqError", "lib", "KVQ_PTR_DEVICE", "KVQ_PTR_HOST_MAPPED",
           "LIBRARY_PATH"]

LIBRARY_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")
KVQ_OK, KVQ_EINVAL, KVQ_ECUDA = 0, -1, -2
KVQ_ETIMEOUT = -1000  # the binding's own: a kernel's status word was set (not a C status)

_i64, _i32, _p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
_LIB = None


class KvqError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        what = ("an internal wait of the kernel timed out; the output is undefined"
                if status == KVQ_ETIMEOUT else lib().kvq_strerror(status).decode())
        super().__init__(f"{name} failed: {what} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libkvq.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIBRARY_PATH):
            raise RuntimeError(
                f"{LIBRARY_PATH} is not built; run `python -m fp8_quantized_paged_store_gb300.build`"
                " or __graft_entry__.build() first")
        L = ctypes.CDLL(LIBRARY_PATH)
        L.kvq_strerror.restype = ctypes.c_char_p
        L.kvq_strerror.argtypes = [ctypes.c_int]
        L.kvq_row_bytes.restype = _i64
        L.kvq_row_bytes.argtypes = [_i64, _i64]
        L.kvq_pointer_kind.restype = ctypes.c_int
        L.kvq_pointer_kind.argtypes = [_p]
        L.kvq_plain_fp8_quotient_mode.restype = ctypes.c_int
        L.kvq_plain_fp8_quotient_mode.argtypes = [ctypes.c_float]
        L.kvq_plain_fp8_checks_run.restype = _i64
        L.kvq_plain_fp8_checks_run.argtypes = []
        L.mxfp4_mla_store.restype = ctypes.c_int
        L.mxfp4_mla_store.argtypes = [_p, _i64, _i64, _i64, _p, _p, _i64, _i64, _i64, _i32, _p]
        L.mxfp4_mla_rmsnorm_store.restype = ctypes.c_int
        L.mxfp4_mla_rmsnorm_store.argtypes = [_p, _i64, _i64, _i64, _p, ctypes.c_float, _p, _p,
                                              _i64, _i64, _i64, _i32, _p]
        for name in ("rope_quant_insert_mxfp8", "rope_quant_insert_nvfp4",
                     "rope_quant_insert_v4"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [_p, _i64, _i64, _p, _p, _i64, _i64, _p, _p, _i64, _i64, _i64, _i32, _i32,
                          _p]
        L.rope_plain_insert.restype = ctypes.c_int
        L.rope_plain_insert.argtypes = [_p, _i64, _i64, _p, _p, _i64, _i64, _p, _p, _i64, _i64,
                                        _i64, _i64, _i32, _i32, ctypes.c_float, _p]
        L.fused_save_compress_norm.restype = ctypes.c_int
        L.fused_save_compress_norm.argtypes = [_p, _i64, _i64, _p, _p, _i32, _p, _p, _i64, _p,
                                               _i64, _i64, _i64, _i64, _p, ctypes.c_float, _p,
                                               _i64, _i64, _p, _p, _i64, _p]
        L.save_ring_rows.restype = ctypes.c_int
        L.save_ring_rows.argtypes = [_p, _i64, _i64, _p, _p, _i64, _i64, _i64, _i64, _p]
        L.mxfp4_mla_gather_dequant.restype = ctypes.c_int
        L.mxfp4_mla_gather_dequant.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _i64, _p, _i64, _p]
        L.mxfp4_mla_sparse_attention.restype = ctypes.c_int
        L.mxfp4_mla_sparse_attention.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _i64, _i64, _i64,
                                                 _p, _i64, ctypes.c_float, _p, _i64, _i64, _p, _p,
                                                 _p, _i64, _p]
        L.mxfp4_mla_sparse_attention_noalloc.restype = ctypes.c_int
        L.mxfp4_mla_sparse_attention_noalloc.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _i64,
                                                         _i64, _i64, _p, _i64, ctypes.c_float, _p,
                                                         _i64, _i64, _p, _p, _p]
        L.mxfp4_mla_sparse_attention_ragged.restype = ctypes.c_int
        L.mxfp4_mla_sparse_attention_ragged.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _i64, _i64,
                                                        _i64, _p, _i64, _p, ctypes.c_float, _p,
                                                        _i64, _i64, _p, _p, _p]
        L.mxfp4_mla_sparse_attention_workspace_size.restype = _i64
        L.mxfp4_mla_sparse_attention_workspace_size.argtypes = [_i64, _i64, _i64]
        _LIB = L
    return _LIB


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _check(name, status):
    if status != KVQ_OK:
        raise KvqError(name, status)


def _device(name, tensors, stream=None):
    """The index of the one CUDA device that every CUDA tensor in `tensors`
    (and a torch stream, if given) lives on, or None when all are pinned host
    tensors. Kernels run on the current device and take raw pointers, so a
    tensor of another GPU would be an illegal address there: raise instead."""
    dev = None
    for t in tensors:
        if t is None or not t.is_cuda:
            continue
        i = t.device.index if t.device.index is not None else torch.cuda.current_device()
        if dev is None:
            dev = i
        elif i != dev:
            raise TypeError(f"{name}: tensors on cuda:{dev} and cuda:{i}; all CUDA arguments must "
                            "be on one device")
    if isinstance(stream, torch.cuda.Stream) and dev is not None and stream.device.index != dev:
        raise TypeError(f"{name}: the stream belongs to cuda:{stream.device.index}, the tensors "
                        f"to cuda:{dev}")
    return dev


def _launch(name, tensors, stream, call):
    """Run `call(stream_handle)` with the tensors' device current (so the
    default stream is that device's) and raise on a nonzero status."""
    dev = _device(name, tensors, stream)
    with torch.cuda.device(dev) if dev is not None else contextlib.nullcontext():
        _check(name, call(_stream(stream)))


KVQ_PTR_DEVICE, KVQ_PTR_HOST_MAPPED = 1, 2


def _host_mapped(t: torch.Tensor) -> bool:
    """A CPU tensor in page-locked memory that the device addresses at the
    same pointer (the library checks; pageable memory never qualifies)."""
    try:
        pinned = t.is_pinned()
    except RuntimeError:
        return False
    if not pinned or t.numel() == 0:
        return False
    return lib().kvq_pointer_kind(t.data_ptr()) == KVQ_PTR_HOST_MAPPED


def _need(t: torch.Tensor, dtype, what):
    """A CUDA tensor of `dtype`, or a pinned CPU one the device addresses."""
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or \
            not (t.is_cuda or (t.device.type == "cpu" and _host_mapped(t))):
        raise TypeError(f"{what} must be a CUDA {dtype} tensor, or a pinned CPU one mapped "
                        f"into the device's address space")


def row_bytes(latent_dim: int = 512, group: int = 32) -> int:
    return int(lib().kvq_row_bytes(latent_dim, group))


def cache_view(cache: torch.Tensor, pitch: int):
    """(num_blocks, block_size, block_stride_rows) of a uint8 cache: either a
    paged [num_blocks, block_size, pitch] view whose rows are contiguous and
    whose block stride is a whole number of rows, or any contiguous tensor
    read as [numel // pitch, pitch] (one block)."""
    _need(cache, torch.uint8, "cache")
    if cache.dim() == 3:
        nb, bs, width = cache.shape
        if width != pitch or cache.stride(2) != 1 or cache.stride(1) != pitch or \
                cache.stride(0) % pitch:
            raise ValueError(f"paged cache {tuple(cache.shape)} with strides {cache.stride()} is "
                             f"not a whole number of {pitch}-byte rows per block")
        return nb, bs, cache.stride(0) // pitch
    if not cache.is_contiguous() or cache.numel() % pitch:
        raise ValueError(f"cache of {cache.numel()} bytes is not a contiguous multiple of {pitch}")
    n = cache.numel() // pitch
    return 1, n, n


def mxfp4_mla_store(latent: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor,
                    group: int = 32, stream=None) -> None:
    """latent: bf16 [T, 512] (any row stride), slot_mapping: int64 [T],
    cache: uint8 paged view (see cache_view) of 272-byte rows."""
    _need(latent, torch.bfloat16, "latent")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if latent.dim() != 2 or latent.stride(1) != 1:
        raise ValueError("latent must be [tokens, latent_dim] with unit column stride")
    if slot_mapping.dim() != 1 or slot_mapping.numel() < latent.shape[0] or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous [tokens] tensor")
    nb, bs, bsr = cache_view(cache, row_bytes(latent.shape[1], group))
    _launch("mxfp4_mla_store", (latent, slot_mapping, cache), stream, lambda s: lib().mxfp4_mla_store(
        latent.data_ptr(), latent.shape[0], latent.shape[1], latent.stride(0),
        slot_mapping.data_ptr(), cache.data_ptr(), nb, bs, bsr, group, s))


def mxfp4_mla_rmsnorm_store(latent: torch.Tensor, weight: torch.Tensor, eps: float,
                            slot_mapping: torch.Tensor, cache: torch.Tensor, group: int = 32,
                            stream=None) -> None:
    """RMSNorm of each latent row (bf16 weight [512], fp32 eps), then the
    MXFP4 store, in one pass; arguments otherwise as mxfp4_mla_store."""
    _need(latent, torch.bfloat16, "latent")
    _need(weight, torch.bfloat16, "weight")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if latent.dim() != 2 or latent.stride(1) != 1:
        raise ValueError("latent must be [tokens, latent_dim] with unit column stride")
    if weight.shape != (latent.shape[1],) or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous [latent_dim] tensor")
    if slot_mapping.dim() != 1 or slot_mapping.numel() < latent.shape[0] or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous [tokens] tensor")
    nb, bs, bsr = cache_view(cache, row_bytes(latent.shape[1], group))
    _launch("mxfp4_mla_rmsnorm_store", (latent, weight, slot_mapping, cache), stream,
            lambda s: lib().mxfp4_mla_rmsnorm_store(
                latent.data_ptr(), latent.shape[0], latent.shape[1], latent.stride(0),
                weight.data_ptr(), float(eps), slot_mapping.data_ptr(), cache.data_ptr(), nb, bs,
                bsr, group, s))


def _rope_inputs(latent, positions, cos_sin, slot_mapping):
    _need(latent, torch.bfloat16, "latent")
    _need(positions, torch.int64, "positions")
    _need(cos_sin, torch.float32, "cos_sin")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if latent.dim() != 2 or latent.shape[1] != 512 or latent.stride(1) != 1:
        raise ValueError("latent must be [tokens, 512] with unit column stride")
    if cos_sin.dim() != 2 or cos_sin.stride(1) != 1:
        raise ValueError("cos_sin must be [rows, >= 64] with unit column stride")
    n = slot_mapping.numel()
    if n > min(latent.shape[0], positions.numel()) or not slot_mapping.is_contiguous() or \
            not positions.is_contiguous():
        raise ValueError("slot_mapping / positions must be contiguous and cover the tokens")
    return n


def _rope(name, record, latent, positions, cos_sin, kv_cache, slot_mapping, compress_ratio,
          sanitize_nans, stream):
    n = _rope_inputs(latent, positions, cos_sin, slot_mapping)
    _need(kv_cache, torch.uint8, "kv_cache")
    if kv_cache.dim() != 3 or kv_cache.shape[-1] != record or not kv_cache[0].is_contiguous():
        raise ValueError(f"kv_cache must be [pages, cache_block, {record}] with contiguous pages")
    _launch(name, (latent, positions, cos_sin, kv_cache, slot_mapping), stream,
            lambda s: getattr(lib(), name)(
                latent.data_ptr(), n, latent.stride(0), positions.data_ptr(), cos_sin.data_ptr(),
                cos_sin.stride(0), cos_sin.shape[0], kv_cache.data_ptr(), slot_mapping.data_ptr(),
                kv_cache.shape[0], kv_cache.shape[1], kv_cache.stride(0), int(compress_ratio),
                1 if sanitize_nans else 0, s))


def rope_quant_insert_mxfp8(latent, positions, cos_sin, kv_cache, slot_mapping, compress_ratio,
                            sanitize_nans=False, stream=None) -> None:
    """kv_cache: uint8 [pages, cache_block, 528]; a page holds cache_block x 512
    value bytes then cache_block x 16 scale bytes."""
    _rope("rope_quant_insert_mxfp8", 528, latent, positions, cos_sin, kv_cache, slot_mapping,
          compress_ratio, sanitize_nans, stream)


def rope_quant_insert_nvfp4(latent, positions, cos_sin, kv_cache, slot_mapping, compress_ratio,
                            sanitize_nans=False, stream=None) -> None:
    """kv_cache: uint8 [pages, cache_block, 288]; a page holds cache_block x 256
    code bytes then cache_block x 32 scale bytes."""
    _rope("rope_quant_insert_nvfp4", 288, latent, positions, cos_sin, kv_cache, slot_mapping,
          compress_ratio, sanitize_nans, stream)


def rope_quant_insert_v4(latent, positions, cos_sin, kv_cache, slot_mapping, compress_ratio,
                         sanitize_nans=False, stream=None) -> None:
    """kv_cache: uint8 [pages, cache_block, 584]; a page holds cache_block x 576
    value bytes (448 E4M3 | 64 bf16) then cache_block x 8 scale bytes."""
    _rope("rope_quant_insert_v4", 584, latent, positions, cos_sin, kv_cache, slot_mapping,
          compress_ratio, sanitize_nans, stream)


def rope_plain_insert(latent, positions, cos_sin, kv_cache, slot_mapping, compress_ratio,
                      fp8_scale=None, stream=None) -> None:
    """kv_cache: bf16 or float8_e4m3fn [pages, cache_block, 512] with unit last
    stride (page and slot strides free, multiples of 8 elements). An fp8 cache
    needs ``fp8_scale`` (the per-tensor dequantizing factor)."""
    n = _rope_inputs(latent, positions, cos_sin, slot_mapping)
    if kv_cache.dtype == torch.bfloat16:
        fp8, scale = 0, 1.0
    elif kv_cache.dtype == torch.float8_e4m3fn:
        if fp8_scale is None:
            raise ValueError("an fp8 kv_cache needs fp8_scale")
        fp8, scale = 1, float(fp8_scale)
    else:
        raise TypeError(f"kv_cache must be bfloat16 or float8_e4m3fn, got {kv_cache.dtype}")
    if not (kv_cache.is_cuda or (kv_cache.device.type == "cpu" and _host_mapped(kv_cache))):
        raise TypeError("kv_cache must be a CUDA tensor, or a pinned CPU one mapped into the "
                        "device's address space")
    if kv_cache.dim() != 3 or kv_cache.shape[2] != 512 or kv_cache.stride(2) != 1:
        raise ValueError("kv_cache must be [pages, cache_block, 512] with unit last stride")
    _launch("rope_plain_insert", (latent, positions, cos_sin, kv_cache, slot_mapping), stream,
            lambda s: lib().rope_plain_insert(
                latent.data_ptr(), n, latent.stride(0), positions.data_ptr(), cos_sin.data_ptr(),
                cos_sin.stride(0), cos_sin.shape[0], kv_cache.data_ptr(), slot_mapping.data_ptr(),
                kv_cache.shape[0], kv_cache.shape[1], kv_cache.stride(0), kv_cache.stride(1),
                int(compress_ratio), fp8, scale, s))


def save_ring_rows(rows: torch.Tensor, slot_mapping: torch.Tensor, state: torch.Tensor,
                   stream=None) -> None:
    """rows: fp32 [N, >= 1024] (unit column stride; the first 1024 values are
    saved); state: fp32 [blocks, state_block, >= 1024] with unit last stride."""
    _need(rows, torch.float32, "rows")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(state, torch.float32, "state")
    if rows.dim() != 2 or rows.shape[1] < 1024 or rows.stride(1) != 1:
        raise ValueError("rows must be [N, >= 1024] with unit column stride")
    if state.dim() != 3 or state.shape[2] < 1024 or state.stride(2) != 1:
        raise ValueError("state must be [blocks, state_block, >= 1024] with unit last stride")
    if slot_mapping.numel() > rows.shape[0] or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous and cover the rows")
    _launch("save_ring_rows", (rows, slot_mapping, state), stream, lambda s: lib().save_ring_rows(
        rows.data_ptr(), slot_mapping.numel(), rows.stride(0), slot_mapping.data_ptr(),
        state.data_ptr(), state.shape[0], state.shape[1], state.stride(0), state.stride(1), s))


def fused_save_compress_norm(kv_score, positions, state_cache, slot_mapping, query_start_loc,
                             token_to_req_indices, rms_norm_weight, rms_norm_eps: float,
                             compress_ratio: int, latent_out, prev_rows=None,
                             prev_row_indices=None, stream=None) -> None:
    """kv_score: fp32 [tokens, 512 * R] (unit column stride); state_cache: fp32
    [blocks, capacity, >= 1024] with unit last stride (R = 2); slot_mapping,
    positions, query_start_loc [num_reqs + 1] and token_to_req_indices: int64
    contiguous; rms_norm_weight: bf16 [512]; latent_out: bf16 [tokens, 512]
    with unit last stride; prev_rows: fp32 [rows, >= 1024] with
    prev_row_indices int64 [num_reqs], or neither."""
    R = int(compress_ratio)
    _need(kv_score, torch.float32, "kv_score")
    _need(positions, torch.int64, "positions")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(rms_norm_weight, torch.bfloat16, "rms_norm_weight")
    _need(latent_out, torch.bfloat16, "latent_out")
    if kv_score.dim() != 2 or kv_score.shape[1] != 512 * R or kv_score.stride(1) != 1:
        raise ValueError("kv_score must be [tokens, 512 * compress_ratio] with unit column stride")
    if latent_out.dim() != 2 or latent_out.shape[1] != 512 or latent_out.stride(1) != 1:
        raise ValueError("latent_out must be [tokens, 512] with unit column stride")
    if rms_norm_weight.numel() != 512 or not rms_norm_weight.is_contiguous():
        raise ValueError("rms_norm_weight must be a contiguous [512] tensor")
    n = slot_mapping.numel()
    if n > min(kv_score.shape[0], positions.numel(), latent_out.shape[0]) or \
            not slot_mapping.is_contiguous() or not positions.is_contiguous():
        raise ValueError("slot_mapping / positions must be contiguous and cover the tokens")
    qsl = t2r = st = prev = pidx = None
    nreq = nb = cap = sst = srs = nprev = pst = 0
    if R == 2:
        _need(query_start_loc, torch.int64, "query_start_loc")
        _need(token_to_req_indices, torch.int64, "token_to_req_indices")
        _need(state_cache, torch.float32, "state_cache")
        if not query_start_loc.is_contiguous() or not token_to_req_indices.is_contiguous() or \
                token_to_req_indices.numel() < n:
            raise ValueError("query_start_loc / token_to_req_indices must be contiguous")
        if state_cache.dim() != 3 or state_cache.shape[2] < 1024 or state_cache.stride(2) != 1:
            raise ValueError("state_cache must be [blocks, capacity, >= 1024] with unit last stride")
        nreq = query_start_loc.numel() - 1
        qsl, t2r, st = query_start_loc.data_ptr(), token_to_req_indices.data_ptr(), \
            state_cache.data_ptr()
        nb, cap = state_cache.shape[0], state_cache.shape[1]
        sst, srs = state_cache.stride(0), state_cache.stride(1)
        if prev_rows is not None:
            _need(prev_rows, torch.float32, "prev_rows")
            _need(prev_row_indices, torch.int64, "prev_row_indices")
            if prev_rows.dim() != 2 or prev_rows.shape[1] < 1024 or prev_rows.stride(1) != 1:
                raise ValueError("prev_rows must be [rows, >= 1024] with unit column stride")
            if prev_row_indices.numel() < nreq or not prev_row_indices.is_contiguous():
                raise ValueError("prev_row_indices must be contiguous and cover the requests")
            prev, pidx = prev_rows.data_ptr(), prev_row_indices.data_ptr()
            nprev, pst = prev_rows.shape[0], prev_rows.stride(0)
    elif R != 1:
        raise ValueError("compress_ratio must be 1 or 2")
    args = (kv_score, positions, slot_mapping, rms_norm_weight, latent_out) + (
        (query_start_loc, token_to_req_indices, state_cache, prev_rows, prev_row_indices)
        if R == 2 else ())
    _launch("fused_save_compress_norm", args, stream, lambda s: lib().fused_save_compress_norm(
        kv_score.data_ptr(), n, kv_score.stride(0), positions.data_ptr(), slot_mapping.data_ptr(),
        R, qsl, t2r, nreq, st, nb, cap, sst, srs, rms_norm_weight.data_ptr(),
        float(rms_norm_eps), prev, nprev, pst, pidx, latent_out.data_ptr(),
        latent_out.stride(0), s))


def mxfp4_mla_gather_dequant(cache: torch.Tensor, indices: torch.Tensor, out: torch.Tensor = None,
                             latent_dim: int = 512, stream=None) -> torch.Tensor:
    """indices: int64 (any shape, contiguous); returns bf16 [*indices.shape,
    latent_dim] (or fills ``out``, whose last dim has unit stride)."""
    _need(indices, torch.int64, "indices")
    if not indices.is_contiguous():
        raise ValueError("indices must be contiguous")
    nb, bs, bsr = cache_view(cache, row_bytes(latent_dim, 32))
    if out is None:
        out = torch.empty((*indices.shape, latent_dim), dtype=torch.bfloat16,
                          device=indices.device, pin_memory=not indices.is_cuda)
    _need(out, torch.bfloat16, "out")
    flat = out.view(-1, latent_dim) if out.is_contiguous() else out.reshape(-1, latent_dim)
    if flat.data_ptr() != out.data_ptr() or flat.stride(1) != 1:
        raise ValueError("out must be viewable as [num_indices, latent_dim] without a copy")
    _launch("mxfp4_mla_gather_dequant", (cache, indices, out), stream,
            lambda s: lib().mxfp4_mla_gather_dequant(
                cache.data_ptr(), nb, bs, bsr, latent_dim, indices.data_ptr(), indices.numel(),
                out.data_ptr(), flat.stride(0), s))
    return out


def mxfp4_mla_sparse_attention(q: torch.Tensor, cache: torch.Tensor, indices: torch.Tensor,
                               sm_scale: float, out: torch.Tensor = None, lse: torch.Tensor = None,
                               status: torch.Tensor = None, workspace="auto", stream=None):
    """q: bf16 [num_queries, num_heads <= 128, 512] (unit last stride, strides
    multiples of 8); cache: uint8 paged view (see cache_view) of 272-byte rows;
    indices: int64 [num_queries, topk] (contiguous; -1 pads). Returns (out bf16
    [num_queries, num_heads, 512], lse fp32 [num_queries, num_heads] or None).

    ``workspace``: "auto" (default) splits the key tiles evenly over the SMs
    (with a workspace allocated here) when one CTA per (query, value half)
    would leave most SMs idle (few queries; see ``attention_prefers_split``),
    True always splits, False never does, and
    a uint8 device tensor of at least ``attention_workspace_size(...)``
    bytes splits with that workspace.
    ``status``: an int32 device tensor of one element that the kernel sets
    nonzero if an internal wait timed out (the output is then undefined); the
    caller reads it. Without one, a status word is made here and read back
    after the launch (this synchronises the stream) and KvqError is raised
    if it is set."""
    _need(q, torch.bfloat16, "q")
    _need(indices, torch.int64, "indices")
    if q.dim() != 3 or q.shape[2] != 512 or q.stride(2) != 1:
        raise ValueError("q must be [num_queries, num_heads, 512] with unit last stride")
    nq, nh, _ = q.shape
    if indices.dim() != 2 or indices.shape[0] != nq or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous [num_queries, topk] tensor")
    nb, bs, bsr = cache_view(cache, row_bytes(512, 32))
    dev = _device("mxfp4_mla_sparse_attention", (q, cache, indices, out, lse, status), stream)
    cuda_dev = torch.device("cuda", dev if dev is not None else torch.cuda.current_device())
    if out is None:
        out = torch.empty((nq, nh, 512), dtype=torch.bfloat16, device=q.device,
                          pin_memory=not q.is_cuda)
    _need(out, torch.bfloat16, "out")
    if out.dim() != 3 or tuple(out.shape) != (nq, nh, 512) or out.stride(2) != 1:
        raise ValueError("out must be [num_queries, num_heads, 512] with unit last stride")
    if lse is not None:
        _need(lse, torch.float32, "lse")
        if tuple(lse.shape) != (nq, nh) or not lse.is_contiguous():
            raise ValueError("lse must be a contiguous [num_queries, num_heads] tensor")
    own_status = status is None
    with torch.cuda.device(cuda_dev):
        if own_status:
            status = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
        _need(status, torch.int32, "status")
        if isinstance(workspace, str):
            if workspace != "auto":
                raise ValueError('workspace must be "auto", True, False or a uint8 tensor')
            workspace = attention_prefers_split(nq, indices.shape[1], cuda_dev)
        if workspace is True:
            nbytes = attention_workspace_size(nq, nh, indices.shape[1])
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=cuda_dev) \
                if nbytes > 0 else None
        elif workspace is False:
            workspace = None
        if workspace is not None:
            _need(workspace, torch.uint8, "workspace")
    _launch("mxfp4_mla_sparse_attention", (q, cache, indices, out, lse, status, workspace), stream,
            lambda s: lib().mxfp4_mla_sparse_attention(
                q.data_ptr(), nq, nh, q.stride(0), q.stride(1), cache.data_ptr(), nb, bs, bsr,
                indices.data_ptr(), indices.shape[1], float(sm_scale), out.data_ptr(),
                out.stride(0), out.stride(1), lse.data_ptr() if lse is not None else None,
                status.data_ptr(), workspace.data_ptr() if workspace is not None else None,
                workspace.numel() if workspace is not None else 0, s))
    if own_status and int(status.item()) != 0:
        raise KvqError("mxfp4_mla_sparse_attention", KVQ_ETIMEOUT)
    return out, lse


def mxfp4_mla_sparse_attention_ragged(q: torch.Tensor, cache: torch.Tensor,
                                      indices: torch.Tensor, key_offsets: torch.Tensor,
                                      sm_scale: float, out: torch.Tensor = None,
                                      lse: torch.Tensor = None, status: torch.Tensor = None,
                                      stream=None):
    """Sparse attention over ragged index runs (sparse prefill): query n uses
    indices[key_offsets[n]:key_offsets[n + 1]] of a flat int64 tensor.
    q: bf16 [num_queries, num_heads <= 128, 512] as for
    mxfp4_mla_sparse_attention; key_offsets: int64 [num_queries + 1],
    contiguous, on the device. Returns (out, lse); ``status`` as there."""
    _need(q, torch.bfloat16, "q")
    _need(indices, torch.int64, "indices")
    _need(key_offsets, torch.int64, "key_offsets")
    if q.dim() != 3 or q.shape[2] != 512 or q.stride(2) != 1:
        raise ValueError("q must be [num_queries, num_heads, 512] with unit last stride")
    nq, nh, _ = q.shape
    if indices.dim() != 1 or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous 1-D tensor")
    if tuple(key_offsets.shape) != (nq + 1,) or not key_offsets.is_contiguous():
        raise ValueError("key_offsets must be a contiguous [num_queries + 1] tensor")
    nb, bs, bsr = cache_view(cache, row_bytes(512, 32))
    dev = _device("mxfp4_mla_sparse_attention_ragged",
                  (q, cache, indices, key_offsets, out, lse, status), stream)
    cuda_dev = torch.device("cuda", dev if dev is not None else torch.cuda.current_device())
    if out is None:
        out = torch.empty((nq, nh, 512), dtype=torch.bfloat16, device=q.device,
                          pin_memory=not q.is_cuda)
    _need(out, torch.bfloat16, "out")
    if out.dim() != 3 or tuple(out.shape) != (nq, nh, 512) or out.stride(2) != 1:
        raise ValueError("out must be [num_queries, num_heads, 512] with unit last stride")
    if lse is not None:
        _need(lse, torch.float32, "lse")
        if tuple(lse.shape) != (nq, nh) or not lse.is_contiguous():
            raise ValueError("lse must be a contiguous [num_queries, num_heads] tensor")
    own_status = status is None
    if own_status:
        with torch.cuda.device(cuda_dev):
            status = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    _need(status, torch.int32, "status")
    _launch("mxfp4_mla_sparse_attention_ragged", (q, cache, indices, key_offsets, out, lse, status),
            stream, lambda s: lib().mxfp4_mla_sparse_attention_ragged(
                q.data_ptr(), nq, nh, q.stride(0), q.stride(1), cache.data_ptr(), nb, bs, bsr,
                indices.data_ptr() if indices.numel() else None, indices.numel(),
                key_offsets.data_ptr(), float(sm_scale), out.data_ptr(), out.stride(0),
                out.stride(1), lse.data_ptr() if lse is not None else None, status.data_ptr(), s))
    if own_status and int(status.item()) != 0:
        raise KvqError("mxfp4_mla_sparse_attention_ragged", KVQ_ETIMEOUT)
    return out, lse


def attention_workspace_size(num_queries: int, num_heads: int, topk: int) -> int:
    """Workspace bytes mxfp4_mla_sparse_attention needs to split these shapes
    over the current device's SMs (0: nothing to split)."""
    n = int(lib().mxfp4_mla_sparse_attention_workspace_size(num_queries, num_heads, topk))
    if n < 0:
        raise KvqError("mxfp4_mla_sparse_attention_workspace_size", n)
    return n


def attention_prefers_split(num_queries: int, topk: int, device=None) -> bool:
    """Whether to split the key tiles over the SMs on this device: whenever
    the library would (its workspace size is nonzero: the 2 x num_queries
    (query, value half) units fill at most half of the SMs and each has at
    least eight 32-key tiles). Measured on a GB300 (128 heads, 2048 keys) the
    split is 3.0x faster than one CTA per unit for one query, 3.0x for four,
    2.0x for sixteen and 1.4x for 32."""
    if topk <= 0 or num_queries <= 0:
        return False
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        return lib().mxfp4_mla_sparse_attention_workspace_size(num_queries, 1, topk) > 0
