"""Pins for the oracle's QUEST block selection and sparse attention."""
import math

import numpy as np
import pytest
import torch

from tests.conftest import golden
from tests.test_oracle_attention import _bits, _paged_from_contiguous


def test_hand_worked_example(oracle_mod):
    g = golden("t7_quest_hand_example.json")
    bs, D = g["block_size"], g["head_dim"]
    keys = torch.tensor(g["keys"]).half()
    NB = 6
    kc = torch.zeros(NB, 1, bs, D).half()
    for pos in range(g["context_len"]):
        kc[g["block_table"][pos // bs], 0, pos % bs] = keys[pos]
    q = torch.tensor([[g["q"]]]).half()
    table = np.array([g["block_table"]], np.int32)
    sel, lens, bounds = oracle_mod.quest_select(_bits(q), 0, _bits(kc), 0, table,
                                                np.array([g["context_len"]], np.int32), g["budget_blocks"])
    assert list(bounds[0, 0]) == g["expected_bounds"]
    assert list(sel[0, 0]) == g["expected_selected_physical"]
    assert lens[0, 0] == g["expected_selected_tokens"]


@pytest.mark.parametrize("G", [1, 4])
def test_bound_dominates_every_key(oracle_mod, G):
    rng = np.random.default_rng(G)
    B, Hkv, D, bs = 3, 2, 32, 8
    lens = np.array([1, 29, 64])
    k = torch.from_numpy(rng.standard_normal((B, Hkv, 64, D))).to(torch.bfloat16)
    q = torch.from_numpy(rng.standard_normal((B, Hkv * G, D))).to(torch.bfloat16)
    kp, vp, tables = _paged_from_contiguous(k, k, lens, bs, rng)
    sel, slen, bounds = oracle_mod.quest_select(_bits(q), 1, _bits(kp), 1, tables, lens.astype(np.int32), 2)
    for b in range(B):
        for h in range(Hkv):
            for j in range(-(-int(lens[b]) // bs)):
                keys = k[b, h, j * bs: min((j + 1) * bs, int(lens[b]))].double().numpy()
                qs = q[b, h * G:(h + 1) * G].double().numpy()
                true_max = float((qs @ keys.T).max())
                assert bounds[b, h, j] >= true_max - 1e-9


def test_budget_covering_all_blocks_is_full_attention(oracle_mod):
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D, bs = 3, 8, 2, 64, 16
    lens = np.array([5, 100, 161])
    k = torch.from_numpy(rng.standard_normal((B, Hkv, 161, D))).half()
    v = torch.from_numpy(rng.standard_normal((B, Hkv, 161, D))).half()
    q = torch.from_numpy(rng.standard_normal((B, Hq, D))).half()
    kp, vp, tables = _paged_from_contiguous(k, v, lens, bs, rng)
    sel, slen, _ = oracle_mod.quest_select(_bits(q), 0, _bits(kp), 0, tables, lens.astype(np.int32), 64)
    assert np.array_equal(slen, np.repeat(lens[:, None], Hkv, axis=1))
    for b in range(B):
        for h in range(Hkv):
            n = -(-int(lens[b]) // bs)
            assert list(sel[b, h, :n]) == list(tables[b, :n])
    got = oracle_mod.sparse_decode(_bits(q), 0, _bits(kp), _bits(vp), 0, sel, slen, 0.125)
    want = oracle_mod.paged_decode(_bits(q), 0, _bits(kp), _bits(vp), 0, tables, lens.astype(np.int32), 0.125)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


def test_planted_key_block_is_selected(oracle_mod):
    rng = np.random.default_rng(2)
    D, bs, L = 32, 16, 16 * 20
    k = torch.from_numpy(rng.standard_normal((1, 1, L, D)) * 0.1).half()
    q = torch.from_numpy(rng.standard_normal((1, 1, D))).half()
    k[0, 0, 7 * 16 + 3] = (q[0, 0].float() * 20).half()  # one key far better aligned with q
    kp, vp, tables = _paged_from_contiguous(k, k, np.array([L]), bs, rng)
    sel, slen, bounds = oracle_mod.quest_select(_bits(q), 0, _bits(kp), 0, tables, np.array([L], np.int32), 1)
    assert sel[0, 0, 0] == tables[0, 7] and slen[0, 0] == 16
    assert int(np.argmax(bounds[0, 0, :20])) == 7


def test_sparse_decode_matches_sdpa_on_selected_tokens(oracle_mod):
    rng = np.random.default_rng(4)
    B, Hq, Hkv, D, bs = 2, 4, 2, 32, 8
    lens = np.array([70, 41])
    k = torch.from_numpy(rng.standard_normal((B, Hkv, 70, D))).half()
    v = torch.from_numpy(rng.standard_normal((B, Hkv, 70, D))).half()
    q = torch.from_numpy(rng.standard_normal((B, Hq, D))).half()
    kp, vp, tables = _paged_from_contiguous(k, v, lens, bs, rng)
    sel, slen, bounds = oracle_mod.quest_select(_bits(q), 0, _bits(kp), 0, tables, lens.astype(np.int32), 3)
    got = oracle_mod.sparse_decode(_bits(q), 0, _bits(kp), _bits(vp), 0, sel, slen, 0.2)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            # logical blocks chosen: the 3 largest bounds, lower index on ties
            n = -(-int(lens[b]) // bs)
            order = sorted(range(n), key=lambda j: (-bounds[b, h, j], j))[:3]
            toks = [t for j in sorted(order) for t in range(j * bs, min((j + 1) * bs, int(lens[b])))]
            assert slen[b, h] == len(toks)
            kk = k[b, h, toks].double()[None].expand(G, -1, -1)
            vv = v[b, h, toks].double()[None].expand(G, -1, -1)
            qq = q[b, h * G:(h + 1) * G].double()[:, None]
            want = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=0.2)[:, 0].numpy()
            np.testing.assert_allclose(got[b, h * G:(h + 1) * G], want, rtol=0, atol=1e-12)


def test_minmax_matches_hand_example(oracle_mod):
    g = golden("t7_quest_hand_example.json")
    bs, D = g["block_size"], g["head_dim"]
    keys = torch.tensor(g["keys"]).half()
    kc = torch.zeros(6, 1, bs, D).half()
    for pos in range(g["context_len"]):
        kc[g["block_table"][pos // bs], 0, pos % bs] = keys[pos]
    mn, mx = oracle_mod.quest_block_minmax(_bits(kc), 0, np.array([g["block_table"]], np.int32),
                                           np.array([g["context_len"]], np.int32))
    assert mn[0, :, 0].tolist() == g["expected_min"] and mx[0, :, 0].tolist() == g["expected_max"]


def _e4m3_paged(rng, B, Hkv, L, D, bs):
    codes = torch.from_numpy(rng.integers(0, 256, size=(B, Hkv, L, D), dtype=np.uint8))
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    kp, _, tables = _paged_from_contiguous(codes, codes, np.full(B, L), bs, rng)
    return codes, kp, tables


def test_e4m3_bound_dominates_every_dequantised_key(oracle_mod):
    """Over an E4M3 cache the bound covers q . (code x k_scale) for every key
    of the block, the codes decoded by torch's float8_e4m3fn."""
    rng = np.random.default_rng(31)
    B, Hkv, G, D, bs, L, ks = 2, 2, 4, 32, 8, 45, 0.0137
    codes, kp, tables = _e4m3_paged(rng, B, Hkv, L, D, bs)
    q = torch.from_numpy(rng.standard_normal((B, Hkv * G, D))).to(torch.bfloat16)
    lens = np.full(B, L, np.int32)
    _, _, bounds = oracle_mod.quest_select(_bits(q), 1, kp.numpy(), 2, tables, lens, 2, k_scale=ks)
    vals = codes.view(torch.float8_e4m3fn).double() * ks
    for b in range(B):
        for h in range(Hkv):
            for j in range(-(-L // bs)):
                keys = vals[b, h, j * bs: min((j + 1) * bs, L)].numpy()
                qs = q[b, h * G:(h + 1) * G].double().numpy()
                assert bounds[b, h, j] >= float((qs @ keys.T).max()) - 1e-9


def test_e4m3_selection_does_not_depend_on_the_scale(oracle_mod):
    """A positive per-tensor scale multiplies every bound by itself, so the
    selection is the same for any k_scale > 0 (bounds scale exactly in ratio)."""
    rng = np.random.default_rng(32)
    B, Hkv, G, D, bs, L = 3, 2, 2, 64, 16, 300
    codes, kp, tables = _e4m3_paged(rng, B, Hkv, L, D, bs)
    q = torch.from_numpy(rng.standard_normal((B, Hkv * G, D))).to(torch.float16)
    lens = np.full(B, L, np.int32)
    s1, l1, u1 = oracle_mod.quest_select(_bits(q), 0, kp.numpy(), 2, tables, lens, 5, k_scale=1.0)
    s2, l2, u2 = oracle_mod.quest_select(_bits(q), 0, kp.numpy(), 2, tables, lens, 5, k_scale=0.0219)
    assert np.array_equal(s1, s2) and np.array_equal(l1, l2)
    n = -(-L // bs)
    np.testing.assert_allclose(u2[:, :, :n], 0.0219 * u1[:, :, :n], rtol=1e-12, atol=0)


def test_e4m3_minmax_is_the_decoded_codes(oracle_mod):
    """E4M3 metadata: channel-wise min and max of the decoded codes (no scale),
    against torch's float8_e4m3fn decoding."""
    rng = np.random.default_rng(33)
    B, Hkv, D, bs, L = 2, 3, 16, 8, 21
    codes, kp, tables = _e4m3_paged(rng, B, Hkv, L, D, bs)
    mn, mx = oracle_mod.quest_block_minmax(kp.numpy(), 2, tables, np.full(B, L, np.int32))
    vals = codes.view(torch.float8_e4m3fn).double()
    for b in range(B):
        for j in range(-(-L // bs)):
            blk = vals[b, :, j * bs: min((j + 1) * bs, L)]
            np.testing.assert_array_equal(mn[b, j], blk.min(dim=1).values.numpy())
            np.testing.assert_array_equal(mx[b, j], blk.max(dim=1).values.numpy())
