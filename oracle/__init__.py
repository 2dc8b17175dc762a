"""CPU oracle for the MXFP4 / MXFP8 / NVFP4 paged KV-cache store.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg use it to decide what the CUDA library must produce. The
product package never imports it, and it imports nothing from the product.

The arithmetic lives in kvq_oracle.c (plain single-threaded C, binary32 without
fused multiply-add); this module only marshals numpy arrays into it. Every
function takes bf16 data as uint16 bit patterns. Large calls may be split over
host threads by token range (``threads``); the C code itself stays serial, and
tokens with distinct slots write disjoint bytes, so the split cannot change a
result.

Parity status: the E2M1 encoder, the MXFP4 scale, the MXFP4 store, the E4M3
encoder, the NVFP4 division, the RoPE rotation and the gather are pinned by the
tests in tests/test_oracle_pins*.py. The treatment of NaN inputs by the V4.1
inserts (NaN-ignoring amax, NaN kept through the clamp as E4M3 0x7F) is pinned
only by the reading stated in kvq_oracle.c: the pages do not fix it.

Two modules hold float64 oracles of operations whose kernels use
transcendental or reduced-precision arithmetic, checked within derived
bounds rather than bit for bit: attention.py (sparse MLA attention over the
packed cache) and compress.py (fused_save_compress_norm: group pooling,
RMSNorm and the ring save).
"""
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_LIB = None

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_ptr = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_row_bytes.restype = _i64
        L.oracle_row_bytes.argtypes = [_i64, _i64]
        L.oracle_ceil_pow2_exponent.restype = _i32
        L.oracle_ceil_pow2_exponent.argtypes = [ctypes.c_float]
        L.oracle_e2m1_code.restype = ctypes.c_uint8
        L.oracle_e2m1_code.argtypes = [ctypes.c_float]
        for name in ("oracle_e2m1_code_array", "oracle_ceil_pow2_exponent_array",
                     "oracle_mxfp4_scale_exponent_array", "oracle_e4m3_encode_array",
                     "oracle_e4m3_decode_array", "oracle_e2m1_value_array"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [_ptr, _ptr, _i64]
        L.oracle_mxfp4_mla_store.restype = None
        L.oracle_mxfp4_mla_store.argtypes = [_ptr, _i64, _i64, _i64, _ptr, _ptr, _i64, _i64, _i64,
                                             _i32]
        L.oracle_mxfp4_mla_gather_dequant.restype = None
        L.oracle_mxfp4_mla_gather_dequant.argtypes = [_ptr, _i64, _i64, _i64, _i64, _i32, _ptr,
                                                      _i64, _ptr, _i64]
        L.oracle_rmsnorm_rows.restype = None
        L.oracle_rmsnorm_rows.argtypes = [_ptr, _i64, _i64, _ptr, ctypes.c_float, _ptr]
        L.oracle_mxfp4_mla_rmsnorm_store.restype = None
        L.oracle_mxfp4_mla_rmsnorm_store.argtypes = [_ptr, _i64, _i64, _ptr, ctypes.c_float, _ptr,
                                                     _ptr, _i64, _i64, _i64]
        for name in ("oracle_rope_quant_insert_mxfp8", "oracle_rope_quant_insert_nvfp4",
                     "oracle_rope_quant_insert_v4"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _i64, _i64, _ptr, _ptr,
                                         _i64, _i64, _i64, _i32, _i32]
        L.oracle_rope_plain_insert.restype = None
        L.oracle_rope_plain_insert.argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _i64, _i64, _ptr,
                                               _ptr, _i64, _i64, _i64, _i64, _i32, _i32,
                                               ctypes.c_float]
        L.oracle_save_ring_rows.restype = None
        L.oracle_save_ring_rows.argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _i64, _i64, _i64, _i64]
        _LIB = L
    return _LIB


def _addr(a: np.ndarray, byte_offset: int = 0) -> int:
    return a.ctypes.data + byte_offset


def _contig(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _elementwise(fn_name, x, in_dtype, out_dtype):
    x = _contig(x, in_dtype)
    out = np.empty(x.shape, dtype=out_dtype)
    getattr(lib(), fn_name)(_addr(x), _addr(out), x.size)
    return out


# ---------------------------------------------------------------- formats ---

def row_bytes(d: int, group: int = 32) -> int:
    return int(lib().oracle_row_bytes(d, group))


def ceil_pow2_exponent(v) -> np.ndarray:
    return _elementwise("oracle_ceil_pow2_exponent_array", v, np.float32, np.int32)


def mxfp4_scale_exponent(amax) -> np.ndarray:
    return _elementwise("oracle_mxfp4_scale_exponent_array", amax, np.float32, np.int32)


def e2m1_code(x) -> np.ndarray:
    return _elementwise("oracle_e2m1_code_array", x, np.float32, np.uint8)


def e2m1_value(codes) -> np.ndarray:
    return _elementwise("oracle_e2m1_value_array", codes, np.uint8, np.float32)


def e4m3_encode(y) -> np.ndarray:
    return _elementwise("oracle_e4m3_encode_array", y, np.float32, np.uint8)


def e4m3_decode(b) -> np.ndarray:
    return _elementwise("oracle_e4m3_decode_array", b, np.uint8, np.float32)


# ------------------------------------------------------------- threading ---

def _split(n: int, threads: int):
    threads = max(1, min(threads, n)) if n else 1
    step = -(-n // threads) if n else 0
    return [(i, min(n, i + step)) for i in range(0, n, step)] if n else []


def _run_split(n, threads, body):
    ranges = _split(n, threads)
    if len(ranges) <= 1:
        for lo, hi in ranges:
            body(lo, hi)
        return
    with ThreadPoolExecutor(len(ranges)) as ex:
        list(ex.map(lambda r: body(*r), ranges))


def _latent_args(latent: np.ndarray):
    """(base address, row stride in elements, rows, cols) of a 2-D uint16 view."""
    assert latent.dtype == np.uint16 and latent.ndim == 2
    assert latent.strides[1] == 2 and latent.strides[0] % 2 == 0
    return latent.ctypes.data, latent.strides[0] // 2, latent.shape[0], latent.shape[1]


# ------------------------------------------------------------ operations ---

def mxfp4_mla_store(latent: np.ndarray, slot_mapping: np.ndarray, cache: np.ndarray,
                    num_blocks: int, block_size: int, block_stride_rows: int,
                    cache_offset: int = 0, group: int = 32, threads: int = 1) -> None:
    """Quantize rows of ``latent`` (uint16 bf16 bits, [T, d] view, any row
    stride) into ``cache`` (flat uint8 buffer, modified in place) at byte
    ``cache_offset`` onwards, laid out as [num_blocks, block_size, row_bytes]
    with ``block_stride_rows`` rows between blocks."""
    base, stride, T, d = _latent_args(latent)
    slots = _contig(slot_mapping, np.int64)
    assert slots.shape[0] >= T and cache.dtype == np.uint8 and cache.flags.c_contiguous
    assert d % group == 0 and group % 2 == 0 and group <= 1024
    pitch = row_bytes(d, group)
    need = cache_offset + ((num_blocks - 1) * block_stride_rows + block_size) * pitch
    assert num_blocks >= 1 and block_stride_rows >= block_size and need <= cache.nbytes
    L = lib()

    def body(lo, hi):
        L.oracle_mxfp4_mla_store(base + lo * stride * 2, hi - lo, d, stride,
                                 _addr(slots, lo * 8), _addr(cache, cache_offset),
                                 num_blocks, block_size, block_stride_rows, group)
    _run_split(T, threads, body)


def rmsnorm_rows(latent: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """bf16 bits [T, 512] of the normalised rows (the reading in kvq_oracle.c)."""
    base, stride, T, d = _latent_args(latent)
    assert d == 512
    w = _contig(weight, np.uint16)
    assert w.shape == (512,)
    out = np.empty((T, 512), dtype=np.uint16)
    lib().oracle_rmsnorm_rows(base, T, stride, _addr(w), eps, _addr(out))
    return out


def mxfp4_mla_rmsnorm_store(latent: np.ndarray, weight: np.ndarray, eps: float,
                            slot_mapping: np.ndarray, cache: np.ndarray, num_blocks: int,
                            block_size: int, block_stride_rows: int, cache_offset: int = 0,
                            threads: int = 1) -> None:
    """RMSNorm of each row (bf16 weight [512], fp32 eps), then the MXFP4 store."""
    base, stride, T, d = _latent_args(latent)
    assert d == 512
    w = _contig(weight, np.uint16)
    slots = _contig(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    L = lib()

    def body(lo, hi):
        L.oracle_mxfp4_mla_rmsnorm_store(base + lo * stride * 2, hi - lo, stride, _addr(w), eps,
                                         _addr(slots, lo * 8), _addr(cache, cache_offset),
                                         num_blocks, block_size, block_stride_rows)
    _run_split(T, threads, body)


def mxfp4_mla_gather_dequant(cache: np.ndarray, num_blocks: int, block_size: int,
                             block_stride_rows: int, indices: np.ndarray, latent_dim: int = 512,
                             cache_offset: int = 0, group: int = 32, out: np.ndarray = None,
                             threads: int = 1) -> np.ndarray:
    """Return bf16 bits [len(indices), latent_dim] of the dequantized rows."""
    idx = _contig(indices, np.int64).reshape(-1)
    n = idx.shape[0]
    if out is None:
        out = np.empty((n, latent_dim), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.strides[1] == 2
    ostride = out.strides[0] // 2
    L = lib()

    def body(lo, hi):
        L.oracle_mxfp4_mla_gather_dequant(_addr(cache, cache_offset), num_blocks, block_size,
                                          block_stride_rows, latent_dim, group,
                                          _addr(idx, lo * 8), hi - lo,
                                          out.ctypes.data + lo * ostride * 2, ostride)
    _run_split(n, threads, body)
    return out


def _rope_insert(fn_name, latent, positions, cos_sin, cache, cache_slots, num_pages, cache_block,
                 page_stride_bytes, compress_ratio, sanitize, threads):
    base, stride, T, d = _latent_args(latent)
    assert d == 512
    pos = _contig(positions, np.int64)
    slots = _contig(cache_slots, np.int64)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    assert cs.ndim == 2 and cs.shape[1] >= 64
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    assert compress_ratio >= 1
    L = lib()
    fn = getattr(L, fn_name)

    def body(lo, hi):
        fn(base + lo * stride * 2, hi - lo, stride, _addr(pos, lo * 8), _addr(cs), cs.shape[1],
           cs.shape[0], _addr(cache), _addr(slots, lo * 8), num_pages, cache_block,
           page_stride_bytes, compress_ratio, 1 if sanitize else 0)
    _run_split(T, threads, body)


def rope_quant_insert_mxfp8(latent, positions, cos_sin, cache, cache_slots, num_pages,
                            cache_block, page_stride_bytes, compress_ratio, sanitize,
                            threads: int = 1) -> None:
    _rope_insert("oracle_rope_quant_insert_mxfp8", latent, positions, cos_sin, cache, cache_slots,
                 num_pages, cache_block, page_stride_bytes, compress_ratio, sanitize, threads)


def rope_quant_insert_nvfp4(latent, positions, cos_sin, cache, cache_slots, num_pages,
                            cache_block, page_stride_bytes, compress_ratio, sanitize,
                            threads: int = 1) -> None:
    _rope_insert("oracle_rope_quant_insert_nvfp4", latent, positions, cos_sin, cache, cache_slots,
                 num_pages, cache_block, page_stride_bytes, compress_ratio, sanitize, threads)


def rope_quant_insert_v4(latent, positions, cos_sin, cache, cache_slots, num_pages,
                         cache_block, page_stride_bytes, compress_ratio, sanitize,
                         threads: int = 1) -> None:
    """The 584-byte V4 record (reading in kvq_oracle.c)."""
    _rope_insert("oracle_rope_quant_insert_v4", latent, positions, cos_sin, cache, cache_slots,
                 num_pages, cache_block, page_stride_bytes, compress_ratio, sanitize, threads)


def rope_plain_insert(latent, positions, cos_sin, cache, cache_slots, num_pages, cache_block,
                      page_stride, slot_stride, compress_ratio, fp8: bool = False,
                      fp8_scale: float = 1.0, threads: int = 1) -> None:
    """Plain [448 NoPE | 64 RoPE] rows into a bf16 (uint8 buffer of 2-byte
    elements) or fp8 cache; strides in elements."""
    base, stride, T, d = _latent_args(latent)
    assert d == 512
    pos = _contig(positions, np.int64)
    slots = _contig(cache_slots, np.int64)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and compress_ratio >= 1
    L = lib()

    def body(lo, hi):
        L.oracle_rope_plain_insert(base + lo * stride * 2, hi - lo, stride, _addr(pos, lo * 8),
                                   _addr(cs), cs.shape[1], cs.shape[0], _addr(cache),
                                   _addr(slots, lo * 8), num_pages, cache_block, page_stride,
                                   slot_stride, compress_ratio, 1 if fp8 else 0, fp8_scale)
    _run_split(T, threads, body)


def save_ring_rows(rows: np.ndarray, slot_mapping: np.ndarray, state: np.ndarray,
                   num_blocks: int, state_block: int, state_stride: int,
                   state_row_stride: int) -> None:
    """rows: float32 [N, >= 1024] (unit column stride); state: flat float32
    buffer modified in place; strides in floats."""
    assert rows.dtype == np.float32 and rows.ndim == 2 and rows.strides[1] == 4
    slots = _contig(slot_mapping, np.int64)
    assert state.dtype == np.float32 and state.flags.c_contiguous
    lib().oracle_save_ring_rows(rows.ctypes.data, rows.shape[0], rows.strides[0] // 4,
                                _addr(slots), _addr(state), num_blocks, state_block,
                                state_stride, state_row_stride)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))
