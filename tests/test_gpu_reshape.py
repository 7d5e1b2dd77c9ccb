"""GPU write path (pa_reshape_and_cache) against the oracle, bit for bit.

Exhaustive over every 16-bit input pattern for the e4m3 quantising path
(hardware cvt vs the oracle's OCP encoder of the fp32 quotient), slot
skipping and out-of-pool flagging, and strided k/v rows.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import have_gpu
from pa_testutil import host_copy

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]


@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.7])
def test_fp8_quantisation_exhaustive_over_16bit_patterns(src, scale, pa_lib):
    H, D, bs = 2, 128, 16
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.int16)
    T = 65536 // (H * D)
    tdt = torch.bfloat16 if src == "bf16" else torch.float16
    k = torch.from_numpy(bits.copy()).view(tdt).reshape(T, H, D).cuda()
    v = torch.flip(k, dims=[0]).contiguous()
    NB = T // bs
    slots = torch.arange(T, dtype=torch.int64, device="cuda")
    kc = torch.zeros((NB, H, bs, D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    pa_lib.reshape_and_cache(k, v, kc, vc, slots, "fp8", scale, scale * 2)
    kr = np.zeros((NB, H, bs, D), np.uint8)
    vr = np.zeros_like(kr)
    oracle.reshape_and_cache(k.cpu(), v.cpu(), kr, vr, slots.cpu().numpy(), src, "fp8",
                             scale, scale * 2)
    got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    for got, ref, srcv in ((got_k, kr, k), (got_v, vr, v)):
        # NaN inputs: both sides give a NaN code (sign of NaN is not part of the contract)
        nan_in = torch.isnan(srcv.float()).cpu().numpy().reshape(NB, bs, H, D).transpose(0, 2, 1, 3)
        same = got == ref
        assert same[~nan_in].all(), f"{(~same & ~nan_in).sum()} codes differ"
        assert ((got[nan_in] & 0x7F) == 0x7F).all()


def test_16bit_copy_skips_negative_slots_and_flags_out_of_pool(pa_lib):
    T, H, D, NB, bs = 9, 2, 64, 6, 16
    g = torch.Generator(device="cuda").manual_seed(1)
    big = torch.randn((T, 3 * H * D), generator=g, device="cuda").to(torch.float16)
    k = big[:, :H * D].view(T, H, D)          # strided rows (row stride 3*H*D)
    v = big[:, H * D:2 * H * D].view(T, H, D)
    slots = torch.tensor([3, -1, 17, 0, 95, -7, 40, 41, 80], dtype=torch.int64, device="cuda")
    sentinel = torch.full((NB, H, bs, D), -2.5, dtype=torch.float16, device="cuda")
    kc, vc = sentinel.clone(), sentinel.clone()
    assert pa_lib.check_device_error() == 0
    pa_lib.reshape_and_cache(k, v, kc, vc, slots)
    kr, vr = host_copy(sentinel), host_copy(sentinel)
    oracle.reshape_and_cache(k.contiguous().cpu(), v.contiguous().cpu(), kr, vr,
                             slots.cpu().numpy(), "f16", "f16")
    assert np.array_equal(host_copy(kc), kr) and np.array_equal(host_copy(vc), vr)
    slots_bad = slots.clone()
    slots_bad[2] = NB * bs + 3
    pa_lib.reshape_and_cache(k, v, kc, vc, slots_bad)
    assert pa_lib.check_device_error() & pa_lib.DEVERR_SLOT
