"""KV-cache append (mla_kv_append): host-side argument checks (CPU) and
bit-exact parity with the oracle's encoder on the GPU, including the
saturating range, subnormals, NaN, padding slots and bad slots; then the
appended rows read back by the attend kernel."""

import ctypes
import math

import numpy as np
import pytest
import torch

import mla_decode_paged_gb300 as mla
from mla_decode_paged_gb300 import workloads as W
from oracle import mla_oracle as O
from tests._bits import bf16_bits, i32, oracle_args, u8
from tests.parity import assert_bf16_close, assert_lse_close

NULL = ctypes.c_void_p(0)
P16 = ctypes.c_void_p(1 << 20)   # never dereferenced: each case fails validation first


@pytest.fixture(scope="module")
def lib():
    mla.build()
    return mla.library()


@pytest.mark.parametrize("kw,msg", [
    (dict(T=-1), b"negative"),
    (dict(kv_c_stride=504), b"kv_c_row_stride"),
    (dict(kv_c_stride=516), b"kv_c_row_stride"),
    (dict(k_pe_stride=60), b"k_pe_row_stride"),
    (dict(k_scale=0.0), b"k_scale"),
    (dict(k_scale=float("inf")), b"k_scale"),
    (dict(k_scale=-1.0), b"k_scale"),
    (dict(slots=NULL), b"null"),
    (dict(kv=ctypes.c_void_p((1 << 20) + 8)), b"misaligned"),
    (dict(pool_rows=0), b"empty KV pool"),
])
def test_kv_append_rejects_bad_arguments(lib, kw, msg):
    a = dict(kv_c=P16, kv_c_stride=512, k_pe=P16, k_pe_stride=64, slots=P16, T=4, k_scale=0.5, kv=P16,
             pool_rows=100)
    a.update(kw)
    st = lib.mla_kv_append(a["kv_c"], a["kv_c_stride"], a["k_pe"], a["k_pe_stride"], a["slots"], a["T"],
                           a["k_scale"], a["kv"], a["pool_rows"], NULL)
    assert st == mla.MLA_ERR_INVALID
    assert msg in lib.mla_last_error()


def test_kv_append_zero_tokens_is_a_no_op(lib):
    assert lib.mla_kv_append(P16, 512, P16, 64, P16, 0, 0.5, P16, 100, NULL) == mla.MLA_OK


def _tokens(T, seed, spread=True):
    g = torch.Generator().manual_seed(seed)
    kv_c = torch.randn(T, 512, generator=g)
    k_pe = torch.randn(T, 64, generator=g)
    if spread:   # magnitudes from subnormal to beyond the e4m3 range once divided by k_scale
        kv_c = kv_c * torch.exp2(torch.randint(-14, 10, (T, 512), generator=g).float())
        k_pe = k_pe * torch.exp2(torch.randint(-14, 10, (T, 64), generator=g).float())
    return kv_c.to(torch.bfloat16), k_pe.to(torch.bfloat16)


@pytest.mark.gpu
@pytest.mark.parametrize("T,pool,k_scale", [(1, 8, 1.0), (37, 200, 0.8), (3000, 5000, 1.25), (513, 513, 0.0625)])
def test_kv_append_bit_exact(T, pool, k_scale):
    g = torch.Generator().manual_seed(T)
    kv0 = torch.randint(0, 256, (pool, 576), generator=g, dtype=torch.uint8)
    kv_c, k_pe = _tokens(T, seed=T)
    kv_c[0, :3] = torch.tensor([float("nan"), float("inf"), -float("inf")]).to(torch.bfloat16)
    perm = torch.randperm(pool, generator=g)[:T].to(torch.int64)
    slots = perm.clone()
    slots[::7] = -1                                      # padding tokens are skipped
    kv = kv0.cuda()
    mla.kv_append(kv, kv_c.cuda(), k_pe.cuda(), slots.cuda(), k_scale)
    torch.cuda.synchronize()
    ref = O.kv_append(u8(kv0), bf16_bits(kv_c), bf16_bits(k_pe), slots.numpy(), k_scale)
    assert np.array_equal(u8(kv), ref)
    assert mla.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("k_scale", [1.0, 0.8, 1.25, 1.0 / 3.0, 448.0, 2.0 ** -10])
def test_kv_append_every_bf16_value(k_scale):
    """Every bf16 bit pattern (zeros, subnormals, normals, infinities, NaNs
    of both signs) through the append, against the oracle's IEEE float32
    quotient and e4m3 rounding: 65,536 values as 114 tokens (the last one
    padded with zeros), in two halves of the kernel's units (kv_c and k_pe)."""
    T, pool = 114, 300
    codes = torch.arange(65536, dtype=torch.int32)
    vals = torch.zeros(T * 576, dtype=torch.int32)
    vals[:65536] = codes
    rows = vals.view(T, 576).to(torch.int16).view(torch.bfloat16)
    kv_c, k_pe = rows[:, :512].contiguous(), rows[:, 512:].contiguous()
    g = torch.Generator().manual_seed(3)
    kv0 = torch.randint(0, 256, (pool, 576), generator=g, dtype=torch.uint8)
    slots = torch.randperm(pool, generator=g)[:T].to(torch.int64)
    kv = kv0.cuda()
    mla.kv_append(kv, kv_c.cuda(), k_pe.cuda(), slots.cuda(), k_scale)
    torch.cuda.synchronize()
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns widened by numpy
        ref = O.kv_append(u8(kv0), bf16_bits(kv_c), bf16_bits(k_pe), slots.numpy(), k_scale)
    assert np.array_equal(u8(kv), ref)
    assert mla.device_status() == 0


@pytest.mark.gpu
def test_kv_append_strided_rows_and_bad_slots_flagged():
    T, pool = 64, 100
    big = torch.randn(T, 1024).to(torch.bfloat16)        # kv_c and k_pe as column views of wider rows
    kv_c, k_pe = big[:, :512], big[:, 512:576]
    kv0 = torch.zeros(pool, 576, dtype=torch.uint8)
    slots = torch.arange(T, dtype=torch.int64)
    slots[5] = pool + 3                                  # out of the pool: skipped and flagged
    kv = kv0.cuda()
    mla.kv_append(kv, big.cuda()[:, :512], big.cuda()[:, 512:576], slots.cuda(), 0.5)
    torch.cuda.synchronize()
    assert mla.device_status() & mla.DEV_BAD_PAGE
    s_ok = slots.clone()
    s_ok[5] = -1
    ref = O.kv_append(u8(kv0), bf16_bits(kv_c.contiguous()), bf16_bits(k_pe.contiguous()), s_ok.numpy(), 0.5)
    assert np.array_equal(u8(kv), ref)
    assert mla.device_status() == 0


@pytest.mark.gpu
def test_appended_tokens_are_attended():
    """Write a batch's last tokens with the append kernel, then run the
    decode step over the cache: parity with the oracle on the same bytes."""
    inp = W.make_inputs(1, "cpu", lengths=[40, 300, 129])
    kv = inp.kv.clone()
    lens = i32(inp.lengths)
    indptr = i32(inp.indptr)
    # each request's last 3 pages receive fresh tokens
    slots = torch.from_numpy(np.concatenate([i32(inp.pages)[indptr[r + 1] - 3:indptr[r + 1]]
                                             for r in range(len(lens))]).astype(np.int64))
    kv_c, k_pe = _tokens(slots.numel(), seed=5, spread=False)
    kv_d = kv.cuda()
    mla.kv_append(kv_d, kv_c.cuda(), k_pe.cuda(), slots.cuda(), inp.kv_scale)
    torch.cuda.synchronize()
    new_kv = O.kv_append(u8(kv), bf16_bits(kv_c), bf16_bits(k_pe), slots.numpy(), inp.kv_scale)
    assert np.array_equal(u8(kv_d), new_kv)
    q, pages, ip = inp.q.cuda(), inp.pages.cuda(), inp.indptr.cuda()
    ns, st = 4, 64
    o, lse = mla.attend(q, kv_d, pages, ip, inp.scale, inp.kv_scale, ns, st, heads=inp.heads)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    a = oracle_args(inp)
    a["kv_codes"] = new_kv
    rlat, rlse = O.attend(**a)
    assert_lse_close(lse_m, rlse, "lse after append")
    assert_bf16_close(latent, rlat, "latent after append")
    assert mla.device_status() == 0
