"""Pins for the float64 paged-attention oracle.

The oracle is checked against what does not depend on it:
* contiguous attention computed by torch's scaled_dot_product_attention in
  float64 on the unpaged keys/values, with the pages scattered by a random
  block permutation (the model sees a contiguous sequence whatever the
  physical placement: OptiVerse "Paged KV cache", section "Block table and
  non-contiguous allocation");
* closed forms: one token gives v_0; equal keys or a zero scale give the mean
  of V; one dominant logit gives its value row;
* a brute-force double loop on tiny inputs.
"""
import math

import numpy as np
import pytest
import torch

TORCH_DT = {0: torch.float16, 1: torch.bfloat16}


def _paged_from_contiguous(k, v, lens, bs, rng, extra_blocks=3):
    """Scatter contiguous per-sequence K/V [B, Hkv, Lmax, D] into a shuffled pool."""
    B, Hkv, Lmax, D = k.shape
    nblk = [-(-int(L) // bs) for L in lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB)
    maxb = max(nblk)
    tables = np.zeros((B, maxb), np.int32)
    kp = torch.randn(NB, Hkv, bs, D, dtype=torch.float64).to(k.dtype)  # garbage in unused slots
    vp = torch.randn(NB, Hkv, bs, D, dtype=torch.float64).to(k.dtype)
    o = 0
    for b in range(B):
        for i in range(nblk[b]):
            phys = int(perm[o]); o += 1
            tables[b, i] = phys
            t0, t1 = i * bs, min((i + 1) * bs, int(lens[b]))
            kp[phys, :, : t1 - t0] = k[b, :, t0:t1]
            vp[phys, :, : t1 - t0] = v[b, :, t0:t1]
    return kp, vp, tables


def _bits(t):
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def _sdpa_reference(q, k, v, lens, scale, G):
    """Per-sequence contiguous attention with torch SDPA in float64."""
    B, Hq, D = q.shape
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        L = int(lens[b])
        kk = k[b, :, :L].double().repeat_interleave(G, dim=0)  # [Hq, L, D]
        vv = v[b, :, :L].double().repeat_interleave(G, dim=0)
        qq = q[b].double()[:, None, :]  # [Hq, 1, D]
        out[b] = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)[:, 0]
    return out.numpy()


@pytest.mark.parametrize("dt,B,Hq,Hkv,D,bs", [
    (0, 4, 8, 8, 64, 16),
    (1, 3, 8, 2, 128, 16),
    (1, 2, 4, 1, 64, 32),
    (0, 5, 6, 3, 32, 8),
])
def test_paged_equals_contiguous_sdpa(oracle_mod, dt, B, Hq, Hkv, D, bs):
    rng = np.random.default_rng(1234 + B + D)
    torch.manual_seed(B * 100 + D)
    lens = rng.integers(1, 4 * bs + 7, size=B)
    lens[0] = 1
    Lmax = int(lens.max())
    k = torch.randn(B, Hkv, Lmax, D).to(TORCH_DT[dt])
    v = torch.randn(B, Hkv, Lmax, D).to(TORCH_DT[dt])
    q = torch.randn(B, Hq, D).to(TORCH_DT[dt])
    scale = 1.0 / math.sqrt(D)
    kp, vp, tables = _paged_from_contiguous(k, v, lens, bs, rng)
    got = oracle_mod.paged_decode(_bits(q), dt, _bits(kp), _bits(vp), dt, tables, lens.astype(np.int32), scale)
    want = _sdpa_reference(q, k, v, lens, scale, Hq // Hkv)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_paged_fp8_equals_sdpa_on_dequantised(oracle_mod):
    rng = np.random.default_rng(7)
    B, H, D, bs = 3, 4, 64, 16
    lens = np.array([5, 40, 33])
    k = (torch.randn(B, H, 40, D) * 3).clamp(-448, 448).to(torch.float8_e4m3fn)
    v = (torch.randn(B, H, 40, D) * 3).clamp(-448, 448).to(torch.float8_e4m3fn)
    q = torch.randn(B, H, D).to(torch.bfloat16)
    ks, vs = 0.0125, 0.5
    kp, vp, tables = _paged_from_contiguous(k.view(torch.uint8), v.view(torch.uint8), lens, bs, rng)
    kp = kp.view(torch.float8_e4m3fn) if kp.dtype == torch.uint8 else kp
    got = oracle_mod.paged_decode(_bits(q), 1, kp.view(torch.uint8).numpy(), vp.view(torch.uint8).numpy(), 2,
                                  tables, lens.astype(np.int32), 0.125, k_scale=ks, v_scale=vs)
    want = _sdpa_reference(q, k.double() * ks, v.double() * vs, lens, 0.125, 1)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def _simple_case(oracle_mod, k, v, q, scale, bs=4):
    B, Hkv, L, D = k.shape
    lens = np.full(B, L)
    kp, vp, tables = _paged_from_contiguous(k, v, lens, bs, np.random.default_rng(3))
    return oracle_mod.paged_decode(_bits(q), 0, _bits(kp), _bits(vp), 0, tables, lens.astype(np.int32), scale)


def test_single_token_returns_its_value(oracle_mod):
    torch.manual_seed(0)
    k = torch.randn(2, 3, 1, 16).half()
    v = torch.randn(2, 3, 1, 16).half()
    q = torch.randn(2, 3, 16).half()
    got = _simple_case(oracle_mod, k, v, q, 0.25)
    assert np.array_equal(got, v[:, :, 0].double().numpy())


def test_equal_keys_give_mean_of_values(oracle_mod):
    torch.manual_seed(1)
    k = torch.randn(1, 2, 1, 16).half().expand(1, 2, 11, 16).contiguous()
    v = torch.randn(1, 2, 11, 16).half()
    q = torch.randn(1, 2, 16).half()
    got = _simple_case(oracle_mod, k, v, q, 0.3)
    np.testing.assert_allclose(got, v.double().mean(dim=2).numpy(), rtol=0, atol=1e-14)


def test_zero_scale_gives_mean_of_values(oracle_mod):
    torch.manual_seed(2)
    k = torch.randn(2, 2, 9, 16).half()
    v = torch.randn(2, 2, 9, 16).half()
    q = torch.randn(2, 2, 16).half()
    got = _simple_case(oracle_mod, k, v, q, 0.0)
    np.testing.assert_allclose(got, v.double().mean(dim=2).numpy(), rtol=0, atol=1e-14)


def test_dominant_logit_selects_its_value(oracle_mod):
    torch.manual_seed(3)
    D, L = 16, 13
    q = torch.zeros(1, 1, D); q[0, 0, 0] = 1.0
    k = torch.zeros(1, 1, L, D); k[0, 0, 7, 0] = 8.0
    v = torch.randn(1, 1, L, D).half()
    got = _simple_case(oracle_mod, k.half(), v, q.half(), 10.0)
    # logits are 80 for token 7 and 0 elsewhere: weight of the rest is 12 e^-80
    np.testing.assert_allclose(got[0, 0], v[0, 0, 7].double().numpy(), rtol=0, atol=1e-30)


def test_brute_force_tiny(oracle_mod):
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, bs = 2, 4, 2, 4, 2
    lens = np.array([3, 5])
    k = torch.from_numpy(rng.standard_normal((B, Hkv, 5, D))).half()
    v = torch.from_numpy(rng.standard_normal((B, Hkv, 5, D))).half()
    q = torch.from_numpy(rng.standard_normal((B, Hq, D))).half()
    kp, vp, tables = _paged_from_contiguous(k, v, lens, bs, rng)
    got = oracle_mod.paged_decode(_bits(q), 0, _bits(kp), _bits(vp), 0, tables, lens.astype(np.int32), 0.7)
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            logits = []
            for j in range(lens[b]):
                logits.append(0.7 * sum(float(q[b, h, d]) * float(k[b, kvh, j, d]) for d in range(D)))
            w = [math.exp(x) for x in logits]
            for d in range(D):
                ref = sum(w[j] * float(v[b, kvh, j, d]) for j in range(lens[b])) / sum(w)
                assert abs(got[b, h, d] - ref) < 1e-12


def test_rejects_bad_arguments(oracle_mod):
    q = np.zeros((1, 2, 8), np.uint16)
    kc = np.zeros((4, 2, 4, 8), np.uint16)
    with pytest.raises(ValueError):  # block id outside the pool
        oracle_mod.paged_decode(q, 0, kc, kc, 0, np.array([[9]], np.int32), np.array([3], np.int32), 1.0)
    with pytest.raises(ValueError):  # empty sequence
        oracle_mod.paged_decode(q, 0, kc, kc, 0, np.array([[1]], np.int32), np.array([0], np.int32), 1.0)
    with pytest.raises(ValueError):  # longer than the table covers
        oracle_mod.paged_decode(q, 0, kc, kc, 0, np.array([[1]], np.int32), np.array([5], np.int32), 1.0)
