"""Pins of the oracle's FP8 cache reader (CPU only).

FlashMLA notes, "FP8 KV Cache Quantization and Dequantization" (V32_FP8Sparse, 656
bytes per token): bytes 0-511 the latent as E4M3, bytes 512-527 four float32 scales
(one per 128-element tile), bytes 528-655 the rope part in bf16; dequantisation returns
BF16.  Expected values below are worked out by hand from that layout.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_head_latent_gb300 import workloads as wl


def _token(codes, scales, rope_bf16):
    t = np.zeros(656, dtype=np.uint8)
    t[:512] = codes
    t[512:528] = np.asarray(scales, dtype=np.float32).view(np.uint8)
    t[528:] = torch.tensor(rope_bf16, dtype=torch.bfloat16).view(torch.uint8).numpy()
    return t


def test_e4m3_matches_torch_on_every_code():
    c = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_float(c)
    ref = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])


def test_e4m3_hand_values():
    # 0x38 = 0.0111.000 -> 2^(7-7) = 1; 0x40 -> 2; 0xB8 -> -1; 0x01 -> subnormal 1/8 * 2^-6;
    # 0x7E -> 1.75 * 2^8 = 448 (largest); 0x7F -> NaN.
    v = oracle.e4m3_to_float(np.array([0x38, 0x40, 0xB8, 0x01, 0x7E, 0x7F], dtype=np.uint8))
    assert v[:5].tolist() == [1.0, 2.0, -1.0, 2.0 ** -9, 448.0] and np.isnan(v[5])


def test_each_tile_takes_its_own_scale():
    # Every code 1.0; scales 1, 2, 4, 8 -> element i dequantises to scale[i // 128].
    t = _token(np.full(512, 0x38, dtype=np.uint8), [1.0, 2.0, 4.0, 8.0], [0.5] * 64)
    ckv, kpe = oracle.dequantize_fp8_cache(t.reshape(1, 1, 656))
    assert ckv[0, 0].tolist() == [1.0] * 128 + [2.0] * 128 + [4.0] * 128 + [8.0] * 128
    assert kpe[0, 0].tolist() == [0.5] * 64


def test_product_is_rounded_to_bf16():
    # code 1.75 (0x3E) times scale 1 + 2^-10: 1.75 + 1.75 * 2^-10 in float32, which lies
    # between the bf16 neighbours 1.75 and 1.7578125 (bf16 keeps 8 significant bits) and
    # is nearer to 1.75.  Scale 1 + 2^-7 + 2^-8 gives 1.75 * 1.01171875 = 1.770508...,
    # whose bf16 neighbours are 1.765625 and 1.7734375: nearer the upper one.
    t = _token(np.array([0x3E, 0x3E] + [0] * 510, dtype=np.uint8),
               [1.0 + 2.0 ** -10, 1.0, 1.0, 1.0], [0.0] * 64)
    ckv, _ = oracle.dequantize_fp8_cache(t.reshape(1, 1, 656))
    assert ckv[0, 0, 0] == 1.75
    t2 = _token(np.array([0x3E] + [0] * 511, dtype=np.uint8), [1.0 + 2.0 ** -7 + 2.0 ** -8, 1.0, 1.0, 1.0],
                [0.0] * 64)
    ckv2, _ = oracle.dequantize_fp8_cache(t2.reshape(1, 1, 656))
    assert ckv2[0, 0, 0] == 1.7734375


def test_dequantised_cache_is_close_to_the_quantised_values():
    w = wl.quantize_fp8(wl.make_decode([70, 200], 4, 64, seed=9))
    ckv, kpe = oracle.dequantize_fp8_cache(w.kv_fp8.numpy())
    ref = w.ckv_cache.double().numpy()
    amax = np.abs(ref.reshape(*ref.shape[:-1], 4, 128)).max(axis=-1, keepdims=True)
    err = np.abs(ckv - ref).reshape(*ref.shape[:-1], 4, 128)
    # E4M3 keeps 4 significant bits: error <= 2^-4 of the tile's largest value, plus
    # the bf16 rounding of the product.
    assert np.all(err <= amax * (2.0 ** -4 + 2.0 ** -8))
    assert np.array_equal(kpe, w.kpe_cache.double().numpy())


def test_decode_is_decode_of_the_dequantised_cache():
    w = wl.quantize_fp8(wl.make_decode([70, 1, 130], 4, 16, seed=10))
    qn, qp = w.q_nope.float().numpy(), w.q_pe.float().numpy()
    out, lse = oracle.mla_decode_fp8(qn, qp, w.kv_fp8.numpy(), w.kv_indptr.numpy(), w.kv_indices.numpy(),
                                     w.sm_scale)
    ckv, kpe = oracle.dequantize_fp8_cache(w.kv_fp8.numpy())
    ref_out, ref_lse = oracle.mla_decode(qn, qp, ckv, kpe, w.kv_indptr.numpy(), w.kv_indices.numpy(), w.sm_scale)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


def _scale_by_position_mod_4(kv_fp8):
    ckv, kpe = oracle.mla_oracle.__dict__["_orig_deq"](kv_fp8)
    raw = np.asarray(kv_fp8)
    scales = np.ascontiguousarray(raw[..., 512:528]).view(np.float32)
    vals = oracle.e4m3_to_float(raw[..., :512])
    return vals * scales[..., np.arange(512) % 4], kpe


def test_tile_pin_catches_a_wrong_scale_index(monkeypatch):
    monkeypatch.setitem(oracle.mla_oracle.__dict__, "_orig_deq", oracle.mla_oracle.dequantize_fp8_cache)
    monkeypatch.setattr(oracle, "dequantize_fp8_cache", _scale_by_position_mod_4)
    with pytest.raises(AssertionError):
        test_each_tile_takes_its_own_scale()
