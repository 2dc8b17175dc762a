"""CPU-only checks of the C ABI: the CUDA library builds for sm_103a, loads,
exports every function include/kvq.h declares, and rejects bad arguments on
the host before any CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "kvq.h")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return kvq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == {"kvq_strerror", "kvq_row_bytes", "kvq_pointer_kind",
                          "kvq_plain_fp8_quotient_mode", "kvq_plain_fp8_checks_run",
                          "mxfp4_mla_store",
                          "mxfp4_mla_rmsnorm_store",
                          "rope_quant_insert_mxfp8", "rope_quant_insert_nvfp4",
                          "rope_quant_insert_v4", "rope_plain_insert", "save_ring_rows",
                          "fused_save_compress_norm",
                          "mxfp4_mla_gather_dequant", "mxfp4_mla_sparse_attention",
                          "mxfp4_mla_sparse_attention_workspace_size",
                          "mxfp4_mla_sparse_attention_noalloc",
                          "mxfp4_mla_sparse_attention_ragged"}
    for n in names:
        assert hasattr(L, n), n
    # exported with C linkage from the shared object itself
    lib = ctypes.CDLL(kvq.LIBRARY_PATH)
    for n in names:
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_row_bytes_and_strerror(L):
    assert kvq.row_bytes(512, 32) == 272
    assert L.kvq_row_bytes(1024, 32) == 544
    assert L.kvq_row_bytes(512, 0) == -1 and L.kvq_row_bytes(500, 32) == -1
    assert L.kvq_row_bytes(512, 3) == -1
    assert b"success" in L.kvq_strerror(0)
    assert b"invalid" in L.kvq_strerror(-1) and b"launch" in L.kvq_strerror(-2)
    assert b"unknown" in L.kvq_strerror(7)


# Fake device addresses: never dereferenced, because every case below is
# rejected (or returns for an empty batch) before anything is launched.
A16, A8 = 0x7F0000000000, 0x7F0000001000


def test_store_validation_on_host(L):
    f = L.mxfp4_mla_store
    ok = [A16, 4, 512, 512, A8, A16, 1, 8, 8, 32, None]
    assert f(*[A16, 0, 512, 512, None, None, 1, 8, 8, 32, None]) == 0   # empty batch
    cases = {2: 256, 3: 500, 9: 16}                                      # dim, stride, group
    for i, v in cases.items():
        a = list(ok); a[i] = v
        assert f(*a) == -1, (i, v)
    for i, v in {1: -1, 6: 0, 7: 0, 8: 7, 0: A16 + 2, 4: A8 + 4, 5: A16 + 8, 3: 516}.items():
        a = list(ok); a[i] = v
        assert f(*a) == -1, (i, v)
    a = list(ok); a[0] = None
    assert f(*a) == -1
    a = list(ok); a[6] = 2 ** 62
    assert f(*a) == -1                                                   # view overflows int64


def test_rmsnorm_store_validation_on_host(L):
    f = L.mxfp4_mla_rmsnorm_store
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
    ok = [A16, 4, 512, 512, A16, 1e-6, A8, A16, 1, 8, 8, 32, None]
    empty = list(ok); empty[1] = 0; empty[0] = None
    assert f(*empty) == 0
    for k, v in {4: None, 4.1: A16 + 2, 5: -1.0, 5.1: float("nan"), 5.2: float("inf"),
                 2: 256, 9: 16}.items():
        a = list(ok); a[int(k)] = v
        assert f(*a) == -1, (k, v)


def test_insert_validation_on_host(L):
    for f, rec in ((L.rope_quant_insert_mxfp8, 528), (L.rope_quant_insert_nvfp4, 288),
                   (L.rope_quant_insert_v4, 584)):
        ok = [A16, 4, 512, A8, A16, 64, 10, A16, A8, 2, 64, 64 * rec, 4, 0, None]
        empty = list(ok); empty[1] = 0; empty[0] = None
        assert f(*empty) == 0
        bad = {1: -3, 2: 500, 5: 62, 5.1: 66, 6: 0, 9: 0, 10: 0, 11: 64 * rec - 16,
               11.1: 64 * rec + 8, 12: 0, 13: 2, 0: A16 + 8, 4: A16 + 4, 7: A16 + 1, 3: A8 + 1}
        for k, v in bad.items():
            a = list(ok); a[int(k)] = v
            assert f(*a) == -1, (rec, k, v)


def test_plain_insert_validation_on_host(L):
    f = L.rope_plain_insert
    ok = [A16, 4, 512, A8, A16, 64, 10, A16, A8, 2, 64, 64 * 512, 512, 4, 1, 0.5, None]
    empty = list(ok); empty[1] = 0; empty[0] = None
    assert f(*empty) == 0
    bad = {1: -3, 2: 500, 5: 62, 6: 0, 9: 0, 10: 0, 11: 63 * 512 + 504, 11.1: 64 * 512 + 4,
           12: 504, 12.1: 516, 13: 0, 14: 2, 15: 0.0, 15.1: -1.0, 15.2: float("nan"),
           15.3: float("inf"), 0: A16 + 8, 7: A16 + 8, 3: A8 + 4}
    for k, v in bad.items():
        a = list(ok); a[int(k)] = v
        assert f(*a) == -1, (k, v)
    # a bf16 cache ignores the scale; 0 is accepted there (empty batch: no launch)
    a = list(empty); a[14] = 0; a[15] = 0.0
    assert f(*a) == 0


def test_ring_rows_validation_on_host(L):
    f = L.save_ring_rows
    ok = [A16, 4, 1024, A8, A16, 2, 8, 8 * 1024, 1024, None]
    empty = list(ok); empty[1] = 0; empty[0] = None
    assert f(*empty) == 0
    bad = {1: -1, 2: 1020, 2.1: 1026, 5: 0, 6: 0, 7: 8 * 1024 - 4, 7.1: 8 * 1024 + 2, 8: 1020,
           8.1: 1030, 0: A16 + 4, 4: A16 + 8, 3: A8 + 4}
    for k, v in bad.items():
        a = list(ok); a[int(k)] = v
        assert f(*a) == -1, (k, v)
    a = list(ok); a[0] = None
    assert f(*a) == -1


def test_compress_validation_on_host(L):
    f = L.fused_save_compress_norm
    # kv, T, stride, pos, slots, R, qsl, t2r, nreq, state, nb, cap, sst, srs, w, eps,
    # prev, nprev, pst, pidx, out, ostride, stream
    ok2 = [A16, 4, 1024, A8, A8, 2, A8, A8, 2, A16, 4, 4, 4 * 1024, 1024, A8, 1e-6,
           None, 0, 0, None, A16, 512, None]
    empty = list(ok2); empty[1] = 0; empty[0] = None
    assert f(*empty) == 0
    bad = {5: 3, 5.1: 0, 1: -1, 2: 1020, 2.1: 1026, 21: 500, 21.1: 516, 15: -1.0,
           15.1: float("nan"), 15.2: float("inf"), 8: -1, 10: 0, 11: 0, 13: 1020, 13.1: 1030,
           12: 4 * 1024 - 4, 12.1: 4 * 1024 + 2, 0: A16 + 4, 3: A8 + 4, 4: A8 + 2, 14: A8 + 2,
           20: A16 + 8, 6: None, 7: None, 9: None, 9.1: A16 + 4}
    for k, v in bad.items():
        a = list(ok2); a[int(k)] = v
        assert f(*a) == -1, (k, v)
    a = list(ok2); a[16] = A16                               # prev_rows without indices
    assert f(*a) == -1
    a = list(ok2); a[16], a[17], a[18], a[19] = A16, 3, 1020, A8   # prev row stride < 1024
    assert f(*a) == -1
    a = list(ok2); a[16], a[17], a[18], a[19] = A16 + 4, 3, 1024, A8
    assert f(*a) == -1
    # R = 1 ignores the request and ring arguments (only shapes are checked)
    ok1 = [A16, 4, 512, A8, A8, 1, None, None, 0, None, 0, 0, 0, 0, A8, 1e-6,
           None, 0, 0, None, A16, 512, None]
    e1 = list(ok1); e1[1] = 0
    assert f(*e1) == 0
    for k, v in {2: 508, 2.1: 514, 0: None, 20: None}.items():
        a = list(ok1); a[int(k)] = v
        assert f(*a) == -1, (k, v)


def test_gather_validation_on_host(L):
    f = L.mxfp4_mla_gather_dequant
    ok = [A16, 1, 8, 8, 512, A8, 4, A16, 512, None]
    empty = list(ok); empty[6] = 0; empty[5] = None
    assert f(*empty) == 0
    for k, v in {4: 256, 8: 500, 8.1: 516, 1: 0, 3: 7, 6: -1, 0: A16 + 4, 7: A16 + 2,
                 5: A8 + 2}.items():
        a = list(ok); a[int(k)] = v
        assert f(*a) == -1, (k, v)


def test_attention_validation_on_host(L):
    f = L.mxfp4_mla_sparse_attention
    ok = [A16, 2, 128, 128 * 512, 512, A16, 1, 8, 8, A8, 16, 0.05, A16, 128 * 512, 512, None,
          None, None, 0, None]
    empty = list(ok); empty[1] = 0; empty[0] = None
    assert f(*empty) == 0
    bad = {1: -1, 2: 0, 2.1: 129, 4: 256, 4.1: 516, 3: 12, 6: 0, 7: 0, 8: 7, 10: -1,
           11: -0.5, 11.1: float("nan"), 11.2: float("inf"), 13: 4, 14: 500, 0: A16 + 2,
           5: A16 + 8, 9: A8 + 4, 12: A16 + 8, 15: A16 + 2, 16: A16 + 1}
    for k, v in bad.items():
        a = list(ok); a[int(k)] = v
        assert f(*a) == -1, (k, v)
    a = list(ok); a[0] = None
    assert f(*a) == -1
    # cache rows whose byte offsets leave int64: rejected like the store's
    a = list(ok); a[6] = 1 << 40; a[8] = 1 << 30
    assert f(*a) == -1
    # a workspace that is misaligned or smaller than the query says (2048
    # keys: the two queries' units are cut into chunks)
    need = L.mxfp4_mla_sparse_attention_workspace_size(2, 128, 2048)
    assert need > 0
    a = list(ok); a[10] = 2048; a[17] = A16 + 16; a[18] = need
    assert f(*a) == -1
    a = list(ok); a[10] = 2048; a[17] = A16; a[18] = need - 1
    assert f(*a) == -1


def test_ragged_attention_validation_on_host(L):
    f = L.mxfp4_mla_sparse_attention_ragged
    ok = [A16, 2, 128, 128 * 512, 512, A16, 1, 8, 8, A8, 40, A8 + 0x100, 0.05, A16, 128 * 512, 512,
          None, None, None]
    empty = list(ok); empty[1] = 0; empty[0] = None
    assert f(*empty) == 0
    bad = {1: -1, 2: 0, 2.1: 129, 10: -1, 11: None, 11.1: A8 + 4, 12: float("nan"), 9: A8 + 4,
           0: A16 + 2, 4: 500, 6: 0}
    for k, v in bad.items():
        a = list(ok); a[int(k)] = v
        assert f(*a) == -1, (k, v)
    a = list(ok); a[9] = None                      # indices null with indices to read
    assert f(*a) == -1


def _sms():
    """The SM count the library sees (148 when no GPU is present)."""
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count \
        if torch.cuda.is_available() else 148


def _chunks(units, tiles, sms):
    """Chunks per unit: min(SMs // units, tiles // 4), none empty; 1 below 2."""
    c = min(sms // units, tiles // 4)
    if c < 2:
        return 1
    per = -(-tiles // c)
    return -(-tiles // per)


def test_attention_workspace_size(L):
    """CTAs x heads x (256 bf16 + one fp32 log-sum-exp), CTAs = 2 x queries x
    chunks; 0 when nothing is split (the units fill the SMs, or too few
    tiles); -1 for shapes the attention rejects."""
    g = L.mxfp4_mla_sparse_attention_workspace_size
    assert g(0, 128, 2048) == 0 and g(3, 128, 0) == 0
    assert g(-1, 128, 16) == -1 and g(2, 0, 16) == -1 and g(2, 129, 16) == -1
    assert g(2, 128, -1) == -1
    sms = _sms()
    piece = 128 * (256 * 2 + 4)
    assert g(128, 128, 2048) == 0                      # 256 units fill the SMs
    assert g(1, 128, 32) == 0 and g(1, 64, 1) == 0     # one tile per unit
    # one query of 2048 keys: 64 tiles per half, 16 chunks of four
    assert g(1, 128, 2048) == 2 * 16 * piece
    for nq, nh, topk in ((3, 64, 4096), (5, 128, 700), (20, 128, 2048)):
        tiles = -(-topk // 32)
        c = _chunks(2 * nq, tiles, sms)
        want = 2 * nq * c * nh * (256 * 2 + 4) if c > 1 else 0
        assert g(nq, nh, topk) == want, (nq, nh, topk)


def test_tensors_on_two_devices_are_refused_before_any_launch():
    """Every CUDA argument must be on one device (raw pointers of another GPU
    would be illegal addresses on the launching one); checked before the
    library is called."""
    import types
    import torch
    a = types.SimpleNamespace(is_cuda=True, device=torch.device("cuda", 0))
    b = types.SimpleNamespace(is_cuda=True, device=torch.device("cuda", 1))
    host = types.SimpleNamespace(is_cuda=False, device=torch.device("cpu"))
    calls = []
    with pytest.raises(TypeError):
        kvq._launch("x", (a, host, b), None, lambda s: calls.append(s) or 0)
    assert calls == []
    assert kvq._device("x", (a, host, None, a)) == 0
    assert kvq._device("x", (host,)) is None


def test_binding_has_the_abi_names():
    for n in ("mxfp4_mla_store", "mxfp4_mla_rmsnorm_store", "rope_quant_insert_mxfp8",
              "rope_quant_insert_nvfp4", "rope_quant_insert_v4", "rope_plain_insert",
              "save_ring_rows", "fused_save_compress_norm", "mxfp4_mla_gather_dequant",
              "mxfp4_mla_sparse_attention", "attention_workspace_size"):
        assert callable(getattr(kvq, n))


def test_binding_refuses_pageable_host_tensors():
    """A CPU tensor reaches the library only when it is pinned and mapped at
    the same device address; a pageable one is refused before any call."""
    import torch
    lat = torch.zeros((4, 512), dtype=torch.bfloat16)
    slots = torch.zeros(4, dtype=torch.int64)
    cache = torch.zeros(8 * 272, dtype=torch.uint8)
    with pytest.raises(TypeError):
        kvq.mxfp4_mla_store(lat, slots, cache)
    with pytest.raises(TypeError):
        kvq.mxfp4_mla_gather_dequant(cache, slots)


def test_pointer_kind_host_side(L):
    """kvq_pointer_kind needs no launch: a null pointer is EINVAL; pageable
    host memory is never reported addressable (KVQ_ECUDA where no device is
    present, KVQ_PTR_UNADDRESSABLE where one is)."""
    assert L.kvq_pointer_kind(None) == -1
    buf = ctypes.create_string_buffer(64)
    assert L.kvq_pointer_kind(ctypes.addressof(buf)) in (-2, 0)


def test_fp8_quotient_check_runs_once_per_scale_for_up_to_eight_scales(L):
    """Alternating fp8 scales (layers with different scales) pay the
    exhaustive host check once each, not on every call; a ninth distinct
    scale evicts the oldest answer."""
    scales = [0.01371 + 0.00077 * k for k in range(9)]   # none a power of two, none used elsewhere
    before = L.kvq_plain_fp8_checks_run()
    modes = [L.kvq_plain_fp8_quotient_mode(s) for s in scales[:2]]
    assert L.kvq_plain_fp8_checks_run() - before == 2
    for _ in range(5):
        assert [L.kvq_plain_fp8_quotient_mode(s) for s in scales[:2]] == modes
    assert L.kvq_plain_fp8_checks_run() - before == 2
    for s in scales[:8]:
        L.kvq_plain_fp8_quotient_mode(s)
    assert L.kvq_plain_fp8_checks_run() - before == 8
    for _ in range(3):
        for s in scales[:8]:
            L.kvq_plain_fp8_quotient_mode(s)
    assert L.kvq_plain_fp8_checks_run() - before == 8
    L.kvq_plain_fp8_quotient_mode(scales[8])
    assert L.kvq_plain_fp8_checks_run() - before == 9
    assert L.kvq_plain_fp8_quotient_mode(0.25) == 2          # power of two: no check
    assert L.kvq_plain_fp8_checks_run() - before == 9
