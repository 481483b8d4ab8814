"""Pins of the oracle's FP8-context attention (CPU only).

* The e4m3 decode equals torch's float8_e4m3fn for every finite code.
* With power-of-two scales every dequantised value is exactly a bf16 value, so
  the FP8 oracle must equal the bf16 oracle run on the dequantised cache.
* With arbitrary scales it equals torch SDPA (float64) on the dequantised
  context plus the visible drafts.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.pins import bf16_round, bf16_to_f64, prefix_tuples


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.oracle_e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert np.isnan(got) and np.isnan(ref[c])
        else:
            assert got == ref[c], (c, got, ref[c])


def _case(seed, B=2, W=3, L=3, Hq=4, Hkv=2, D=16, C=40):
    rng = np.random.default_rng(seed)
    beams = rng.integers(0, 3, size=(B, W, L)).astype(np.int32)
    P = W * L
    pk = oracle.oracle_pack(beams, P)
    lens = rng.integers(1, C + 1, size=B)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = bf16_round(rng.standard_normal((B, P, Hq, D)).astype(np.float32))
    kn = bf16_round(rng.standard_normal((B, P, Hkv, D)).astype(np.float32))
    vn = bf16_round(rng.standard_normal((B, P, Hkv, D)).astype(np.float32))
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    kc = rng.choice(finite, size=(offs[-1], Hkv, D)).astype(np.uint8)
    vc = rng.choice(finite, size=(offs[-1], Hkv, D)).astype(np.uint8)
    return beams, pk, q, kn, vn, kc, vc, offs


def _dequant(codes, scale):
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * scale


@pytest.mark.parametrize("ks,vs", [(0.25, 2.0), (1.0 / 64, 1.0 / 8)])
def test_power_of_two_scales_equal_the_bf16_oracle(ks, vs):
    beams, pk, q, kn, vn, kc, vc, offs = _case(1)
    got = oracle.oracle_tree_attention_fp8(q, kn, vn, kc, vc, ks, vs, offs, pk["packed_len"],
                                           pk["mask"])
    kb = bf16_round(_dequant(kc, ks).astype(np.float32))
    vb = bf16_round(_dequant(vc, vs).astype(np.float32))
    assert np.array_equal(bf16_to_f64(kb), _dequant(kc, ks))      # exact in bf16
    ref = oracle.oracle_tree_attention(q, kn, vn, kb, vb, offs, pk["packed_len"], pk["mask"])
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_arbitrary_scales_match_torch_sdpa():
    ks, vs = 0.0123, 0.0371
    beams, pk, q, kn, vn, kc, vc, offs = _case(2, B=1)
    got = oracle.oracle_tree_attention_fp8(q, kn, vn, kc, vc, ks, vs, offs, pk["packed_len"],
                                           pk["mask"])
    P = int(pk["packed_len"][0])
    pref = prefix_tuples(beams[0])
    vis = np.array([[pref[a][: len(pref[k])] == pref[k] for k in range(P)] for a in range(P)])
    C = int(offs[1])
    allowed = np.concatenate([np.ones((P, C), bool), vis], 1)
    Hq, Hkv = q.shape[2], kn.shape[2]
    for hq in range(Hq):
        h = hq // (Hq // Hkv)
        Q = torch.from_numpy(bf16_to_f64(q[0, :P, hq]))
        K = torch.from_numpy(np.concatenate([_dequant(kc[:, h], ks), bf16_to_f64(kn[0, :P, h])]))
        V = torch.from_numpy(np.concatenate([_dequant(vc[:, h], vs), bf16_to_f64(vn[0, :P, h])]))
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[None], K[None], V[None], attn_mask=torch.from_numpy(allowed)[None])[0].numpy()
        np.testing.assert_allclose(got[0, :P, hq], ref, rtol=1e-10, atol=1e-12)
