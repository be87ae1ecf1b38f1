"""CPU checks of the C ABI: the library builds, loads, exports every symbol
the header declares, rejects bad arguments on the host before any launch,
and its split-plan helper is sane.  No kernel runs here."""

import ctypes
import os
import re

import pytest
import torch

import mla_decode_paged_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mla.build()
    return mla.library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ("mla_decode_attend", "mla_merge_splits", "mla_value_gate"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.mla_version()
    assert lib.mla_status_string(0) == b"ok"
    assert lib.mla_status_string(-1) == b"invalid argument"


NULL = ctypes.c_void_p(0)
P16 = ctypes.c_void_p(1 << 20)  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("kw,msg", [
    (dict(qlen=0), b"qlen"),
    (dict(qlen=17), b"qlen"),
    (dict(heads=0), b"heads"),
    (dict(heads=129), b"heads"),
    (dict(num_splits=0), b"num_splits"),
    (dict(num_splits=257), b"num_splits"),
    (dict(split_tokens=0), b"split_tokens"),
    (dict(q_row_stride=12 * 576 - 8), b"q_row_stride"),
    (dict(q_row_stride=12 * 576 + 4), b"q_row_stride"),
    (dict(q=NULL), b"null"),
    (dict(o=NULL), b"null"),
    (dict(q=ctypes.c_void_p((1 << 20) + 8)), b"misaligned"),
    (dict(pool_rows=0), b"empty KV pool"),
    (dict(scale=float("nan")), b"non-finite"),
])
def test_attend_rejects_bad_arguments(lib, kw, msg):
    a = dict(q=P16, q_row_stride=12 * 576, kv=P16, pool_rows=100, pages=P16, num_pages=10, indptr=P16,
             R=2, qlen=1, heads=12, scale=0.1, kv_scale=1.0, num_splits=4, split_tokens=16, o=P16, lse=P16,
             stream=NULL)
    a.update(kw)
    f = lib.mla_decode_attend
    st = f(a["q"], a["q_row_stride"], a["kv"], a["pool_rows"], a["pages"], a["num_pages"], a["indptr"],
           a["R"], a["qlen"], a["heads"], a["scale"], a["kv_scale"], a["num_splits"], a["split_tokens"],
           a["o"], a["lse"], a["stream"])
    assert st == mla.MLA_ERR_INVALID
    assert msg in lib.mla_last_error()


def _attend_ex(lib, flags, **kw):
    a = dict(q=P16, q_row_stride=12 * 576, kv=P16, pool_rows=100, pages=P16, num_pages=10, indptr=P16,
             R=2, qlen=4, heads=12, scale=0.1, kv_scale=1.0, num_splits=4, split_tokens=16, o=P16, lse=P16,
             stream=NULL)
    a.update(kw)
    return lib.mla_decode_attend_ex(a["q"], a["q_row_stride"], a["kv"], a["pool_rows"], a["pages"], a["num_pages"],
                                    a["indptr"], a["R"], a["qlen"], a["heads"], a["scale"], a["kv_scale"],
                                    a["num_splits"], a["split_tokens"], a["o"], a["lse"], flags, a["stream"])


def test_attend_ex_rejects_unknown_flags_and_checks_like_attend(lib):
    # every case below must fail host validation: the pointers are fake
    assert _attend_ex(lib, 4) == mla.MLA_ERR_INVALID
    assert b"flag" in lib.mla_last_error()
    assert _attend_ex(lib, 0x80000000) == mla.MLA_ERR_INVALID
    assert _attend_ex(lib, mla.ATTEND_CAUSAL, qlen=0) == mla.MLA_ERR_INVALID
    assert _attend_ex(lib, mla.ATTEND_CAUSAL, q=NULL) == mla.MLA_ERR_INVALID
    # no requests: nothing to launch
    assert _attend_ex(lib, mla.ATTEND_CAUSAL, R=0) == mla.MLA_OK


@pytest.mark.parametrize("kw,msg", [
    (dict(R=-1), b"num_requests"),
    (dict(qlen=17), b"qlen"),
    (dict(heads=129), b"heads"),
    (dict(num_splits=0), b"num_splits"),
    (dict(split_tokens=0), b"split_tokens"),
    (dict(q_row_stride=12 * 576 + 4), b"q_row_stride"),
    (dict(o=NULL), b"null"),
    (dict(kv=ctypes.c_void_p((1 << 20) + 8)), b"misaligned"),
    (dict(pool_rows=0), b"empty KV pool"),
    (dict(kv_scale=float("inf")), b"non-finite"),
])
def test_warp_mma_cross_check_checks_like_attend(lib, kw, msg):
    """The tests' second attend kernel (mla_debug_attend_mma) refuses the
    arguments mla_decode_attend refuses, before any launch."""
    a = dict(q=P16, q_row_stride=12 * 576, kv=P16, pool_rows=100, pages=P16, num_pages=10, indptr=P16,
             R=2, qlen=1, heads=12, scale=0.1, kv_scale=1.0, num_splits=4, split_tokens=16, o=P16, lse=P16,
             stream=NULL)
    a.update(kw)
    st = lib.mla_debug_attend_mma(a["q"], a["q_row_stride"], a["kv"], a["pool_rows"], a["pages"], a["num_pages"],
                                  a["indptr"], a["R"], a["qlen"], a["heads"], a["scale"], a["kv_scale"],
                                  a["num_splits"], a["split_tokens"], a["o"], a["lse"], a["stream"])
    assert st == (mla.MLA_ERR_UNSUPPORTED if kw.get("pool_rows", 1) > 2**31 else mla.MLA_ERR_INVALID)
    assert msg in lib.mla_last_error()


def test_no_environment_switch_changes_the_attend_kernel(lib, monkeypatch):
    """The product calls always run the tcgen05 kernel: the warp-MMA kernel is
    reachable only through its own test entry point, so options it lacks are
    never refused because of the environment."""
    monkeypatch.setenv("MLA_ATTEND_KERNEL", "mma")
    assert _attend_ex(lib, mla.ATTEND_CAUSAL, R=0) == mla.MLA_OK
    assert _attend_ex(lib, mla.ATTEND_CAUSAL, qlen=0) == mla.MLA_ERR_INVALID
    assert b"qlen" in lib.mla_last_error()


def test_merge_and_value_gate_reject_bad_arguments(lib):
    assert lib.mla_merge_splits(P16, P16, 0, 4, 12, P16, NULL, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_merge_splits(P16, P16, 2, 4, 0, P16, NULL, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_merge_splits(NULL, P16, 2, 4, 12, P16, NULL, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_value_gate(P16, P16, P16, P16, 2, 0, 12, P16, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_value_gate(P16, NULL, P16, P16, 2, 1, 12, P16, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_debug_gather(P16, 10, P16, 5, P16, 1, 6, P16, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_merge_value_gate(P16, P16, 0, P16, P16, P16, 2, 1, 12, P16, NULL, NULL, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_merge_value_gate(P16, P16, 2, NULL, P16, P16, 2, 1, 12, P16, P16, NULL, NULL) == mla.MLA_ERR_INVALID
    assert lib.mla_merge_value_gate(P16, P16, 2, P16, P16, P16, 2, 1, 12, P16, NULL, NULL, NULL) == mla.MLA_ERR_INVALID
    # empty work is a no-op, not an error (and launches nothing)
    assert lib.mla_merge_splits(P16, P16, 2, 0, 12, P16, NULL, NULL) == mla.MLA_OK
    assert lib.mla_value_gate(P16, P16, P16, P16, 0, 1, 12, P16, NULL) == mla.MLA_OK


@pytest.mark.parametrize("R,qlen,H,max_len,total", [
    (2, 1, 12, 100, 164), (64, 1, 12, 8192, 295000), (128, 4, 12, 32768, 2359000),
    (32, 1, 96, 32768, 1 << 20), (256, 8, 12, 131072, 4700000), (1, 1, 12, 1, 1), (8, 16, 128, 500, 2000)])
def test_choose_splits_plan_is_valid(R, qlen, H, max_len, total):
    ns, st = mla.choose_splits(R, qlen, H, max_len, total, sm_count=152)
    assert 1 <= ns <= 256 and st >= 1
    assert -(-max_len // st) <= ns          # the longest request fits in ns splits of st tokens
    if max_len * R >= 1 << 20:
        assert ns >= 2                      # long work is split to fill the SMs
    # with exact host lengths
    lens = [max_len] + [max(0, (total - max_len) // max(1, R - 1))] * (R - 1)
    ns2, st2 = mla.choose_splits(R, qlen, H, sm_count=152, lengths=lens)
    assert 1 <= ns2 <= 256 and -(-max_len // st2) <= ns2


@pytest.mark.parametrize("qlen,H,sms", [(0, 12, 152), (17, 12, 152), (1, 0, 152), (1, 129, 152), (1, 12, 65537)])
def test_choose_splits_rejects_out_of_range_arguments(qlen, H, sms):
    with pytest.raises(mla.MlaError) as e:
        mla.choose_splits(4, qlen, H, 1000, 4000, sm_count=sms)
    assert e.value.status == mla.MLA_ERR_INVALID


def test_binding_rejects_host_tensors_before_any_launch():
    """Host tensors (whose pointers a kernel would fault on) and tensors on
    another device are refused in the binding."""
    q = torch.zeros(2, 12, 576, dtype=torch.bfloat16)
    kv = torch.zeros(8, 576, dtype=torch.uint8)
    pages = torch.zeros(4, dtype=torch.int32)
    indptr = torch.tensor([0, 2, 4], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        mla.attend(q, kv, pages, indptr, 0.1, 1.0, 2, 16)
    o = torch.zeros(2, 2, 12, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        mla.merge(o, torch.zeros(2, 2, 12))
    with pytest.raises(ValueError, match="CUDA tensors"):
        mla.kv_append(kv, torch.zeros(1, 512, dtype=torch.bfloat16), torch.zeros(1, 64, dtype=torch.bfloat16),
                      torch.zeros(1, dtype=torch.int64), 1.0)
    with pytest.raises(ValueError, match="gate is on cpu"):
        mla._same_device(torch.device("cuda", 0), gate=torch.zeros(1))
    with pytest.raises(ValueError, match="o must be a contiguous"):
        mla._buffer(torch.zeros(2, 3), "o", torch.float32, (3, 2))
    with pytest.raises(ValueError, match="o must be a contiguous"):
        mla._buffer(torch.zeros(3, 2).t(), "o", torch.float32, (2, 3))
    mla._buffer(torch.zeros(2, 3), "o", torch.float32, (2, 3))


def test_sm_count_from_a_missing_device_is_an_error(lib):
    """Without a device the host plans cannot take the SM count from it:
    they fail instead of sizing for a guessed grid."""
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    with pytest.raises(mla.MlaError) as e:
        mla.choose_splits(4, 1, 12, 1000, 4000)
    assert e.value.status == mla.MLA_ERR_CUDA
    lens = torch.tensor([100, 200], dtype=torch.int32)
    assert lib.mla_plan_units(2, 1, 12, ctypes.c_void_p(lens.data_ptr()), 4, 0, None, 0, None) == mla.MLA_ERR_CUDA
    assert b"sm_count" in lib.mla_last_error()


def _attend_paged(lib, page_size, last=P16, flags=0, **kw):
    a = dict(q=P16, q_row_stride=12 * 576, kv=P16, pool_rows=128, pages=P16, num_pages=10, indptr=P16,
             R=2, qlen=1, heads=12, scale=0.1, kv_scale=1.0, num_splits=4, split_tokens=16, o=P16, lse=P16,
             stream=NULL)
    a.update(kw)
    return lib.mla_decode_attend_paged(a["q"], a["q_row_stride"], a["kv"], a["pool_rows"], a["pages"],
                                       a["num_pages"], a["indptr"], last, page_size, a["R"], a["qlen"], a["heads"],
                                       a["scale"], a["kv_scale"], a["num_splits"], a["split_tokens"], a["o"],
                                       a["lse"], flags, a["stream"])


@pytest.mark.parametrize("page_size,kw,msg", [
    (0, {}, b"page_size"), (3, {}, b"page_size"), (512, {}, b"page_size"), (24, {}, b"page_size"),
    (16, dict(pool_rows=100), b"multiple of page_size"),
])
def test_attend_paged_rejects_bad_page_arguments(lib, page_size, kw, msg):
    assert _attend_paged(lib, page_size, **kw) == mla.MLA_ERR_INVALID
    assert msg in lib.mla_last_error()


def test_attend_paged_needs_last_page_len(lib):
    assert _attend_paged(lib, 16, last=NULL) == mla.MLA_ERR_INVALID
    assert b"last_page_len" in lib.mla_last_error()
    assert _attend_paged(lib, 16, last=ctypes.c_void_p((1 << 20) + 2)) == mla.MLA_ERR_INVALID


def test_fp8_query_flag_checks(lib):
    # fp8 rows: the stride counts bytes and must be a multiple of 16
    assert _attend_ex(lib, mla.ATTEND_Q_FP8, q_row_stride=12 * 576 + 8) == mla.MLA_ERR_INVALID
    assert b"multiple of 16" in lib.mla_last_error()
    assert _attend_ex(lib, mla.ATTEND_Q_FP8 | 4) == mla.MLA_ERR_INVALID
