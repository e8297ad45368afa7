"""Pins of the oracle's 8-bit KV cache (E4M3 codes with one fp32 scale per row).

The codec is checked against an independent implementation of the format
(torch.float8_e4m3fn), the quantisation against the format's error bound, and the
attention against torch SDPA on K/V that torch decodes, and against the bf16 oracle
when both caches hold the same values.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import (e4m3_probe_values, fp8_append_case, fp8_append_ok, fp8_attention_case,
                          fp8_sdpa_reference, make_case)


def torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(got, torch_decode(codes), equal_nan=True)
    # facts of the format: 1.0, the largest finite, the smallest normal and subnormal, NaN
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.count_nonzero(np.isnan(got)) == 2


def test_e4m3_encode_matches_torch_within_range():
    x = e4m3_probe_values(seed=11, n=20000)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_e4m3_ties_go_to_the_even_mantissa():
    # 1.0625 lies halfway between 1.0 (m=0) and 1.125 (m=1); 1.1875 between m=1 and m=2;
    # 3 * 2^-10 between the subnormals 1 and 2 (x 2^-9); 2^-10 between 0 and 2^-9
    got = oracle.e4m3_encode([1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, -1.0625])
    assert [int(c) for c in got] == [0x38, 0x3A, 0x02, 0x00, 0xB8]


def test_e4m3_saturates_and_keeps_nan_and_signed_zero():
    got = oracle.e4m3_encode([448.5, 464.0, 1e6, float("inf"), -500.0, float("-inf"), float("nan"),
                              -0.0, -1e-9])
    assert [int(c) for c in got] == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80, 0x80]


def test_e4m3_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_fp8_append_places_and_quantises_rows(seed):
    c = fp8_append_case(seed=seed)
    kc, vc, ks, vs = oracle.kv_append_fp8(c["kc"], c["vc"], c["ks"], c["vs"], c["kn"], c["vn"], c["bt"],
                                          c["cu"], c["sl"], block_size=c["bs"])
    assert fp8_append_ok(c, kc, vc, ks, vs)


def test_fp8_append_scale_is_the_row_maximum_over_448():
    c = fp8_append_case(seed=24)
    kc, vc, ks, vs = oracle.kv_append_fp8(c["kc"], c["vc"], c["ks"], c["vs"], c["kn"], c["vn"], c["bt"],
                                          c["cu"], c["sl"], block_size=c["bs"])
    b, slot = c["where"][0]
    for h in range(kc.shape[2]):
        amax = np.float32(np.abs(c["kn"][0, h].float().numpy()).max())
        assert ks[b, h, slot] == np.float32(amax / np.float32(448.0))


@pytest.mark.parametrize("seed,seq_lens,q_lens", [(31, (13, 6, 21), (1, 6, 4)), (32, (1,), (1,)),
                                                  (33, (16, 9), (16, 1))])
def test_fp8_attention_matches_sdpa_on_torch_decoded_kv(seed, seq_lens, q_lens):
    c = fp8_attention_case(seed=seed, seq_lens=seq_lens, q_lens=q_lens)
    out, lse = oracle.attention_fp8(c["q"], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["cu"], c["sl"],
                                    scale=c["scale"])
    ref_out, ref_lse = fp8_sdpa_reference(c)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-12)


def test_fp8_attention_equals_bf16_oracle_on_the_same_values():
    # E4M3 values are exact in bf16: with unit scales both caches hold the same numbers,
    # and the two attentions must agree to the last bit
    c = fp8_attention_case(seed=41)
    ones = np.ones_like(c["ks"])
    out8, lse8 = oracle.attention_fp8(c["q"], c["kc"], c["vc"], ones, ones, c["bt"], c["cu"], c["sl"],
                                      scale=c["scale"])
    kp = torch.from_numpy(torch_decode(c["kc"])).to(torch.bfloat16)
    vp = torch.from_numpy(torch_decode(c["vc"])).to(torch.bfloat16)
    assert np.array_equal(kp.double().numpy(), torch_decode(c["kc"]))
    out16, lse16 = oracle.attention(c["q"], kp, vp, c["bt"], c["cu"], c["sl"], scale=c["scale"])
    assert np.array_equal(out8, out16) and np.array_equal(lse8, lse16)


def test_fp8_attention_of_a_single_key_returns_its_dequantised_v():
    c = fp8_attention_case(seed=42, seq_lens=(1,), q_lens=(1,))
    out, _ = oracle.attention_fp8(c["q"], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["cu"], c["sl"],
                                  scale=c["scale"])
    b = int(c["bt"][0, 0])
    for h in range(c["hq"]):
        g = h // (c["hq"] // c["hkv"])
        v = torch_decode(c["vc"][b, 0, g]) * float(c["vs"][b, g, 0])
        assert np.array_equal(out[0, h], v)
