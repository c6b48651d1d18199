"""Pins of the oracle's number-format decoders and fp8 quantiser against
library routines (numpy float16, torch bfloat16 / float8_e4m3fn), which the
oracle does not use."""
import numpy as np
import pytest
import torch

import oracle


def test_f16_all_codes_match_numpy():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = oracle.f16_to_double(codes)
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


def test_bf16_all_codes_match_torch():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_to_double(codes)
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_double(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 only: the "fn" variant has no infinities
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(got[nan]))
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_encoder_matches_torch_round_to_nearest_even():
    g = torch.Generator().manual_seed(7)
    x = torch.cat([
        torch.randn(20000, generator=g) * 40.0,
        torch.randn(5000, generator=g) * 0.01,            # subnormal range
        torch.rand(2000, generator=g) * 464.0 - 232.0,
    ]).float()
    # exact midpoints between neighbouring codes exercise ties-to-even
    vals = torch.arange(0, 126, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    mids = ((vals[:-1] + vals[1:]) / 2).float()
    x = torch.cat([x, mids, -mids])
    x = x[x.abs() <= 464.0]  # torch turns |x| > 464 into NaN; the oracle saturates
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_from_float(x.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encoder_saturates_and_keeps_sign():
    got = oracle.e4m3_from_float(np.array([465.0, 1e6, np.inf, -1e30, -0.0, 1e-30],
                                          dtype=np.float32))
    assert list(got) == [0x7e, 0x7e, 0x7e, 0xfe, 0x80, 0x00]
    assert oracle.e4m3_from_float(np.array([np.nan], dtype=np.float32))[0] == 0x7f
