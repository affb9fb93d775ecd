"""Prefix caching end to end on the GPU: requests that share a system prompt
reuse its full blocks (their K/V are written once, by the first request), and
decode over the shared blocks matches the float64 oracle computed with the
oracle's own allocator, append and tables."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager_ref import RefBlockManager
from tests.parity import TOL, assert_attention_close, bits

pytestmark = pytest.mark.gpu


def _kv_for_prefix(tokens, pos, Hkv, D):
    """K/V of token `pos`: a deterministic function of tokens[: pos + 1], as in a model."""
    seed = zlib.crc32(np.asarray(tokens[: pos + 1], dtype=np.int32).tobytes())
    rng = np.random.default_rng(seed)
    return rng.standard_normal((2, Hkv, D)).astype(np.float32)


def test_prefix_cached_decode_matches_oracle(pkv_lib, cuda_device):
    pkv = pkv_lib
    pkv.device_error(reset=True)
    bs, Hq, Hkv, D, NB = 16, 8, 4, 64, 64
    rng = np.random.default_rng(3)
    system = list(rng.integers(0, 30000, size=50))  # 3 full blocks + 2 tokens
    prompts = [system + list(rng.integers(0, 30000, size=int(n))) for n in (9, 30, 0, 61)]
    prompts.append(list(rng.integers(0, 30000, size=20)))  # unrelated request
    bm = pkv.BlockManager(NB, bs)
    ref = RefBlockManager(NB, bs)
    kc = torch.zeros(NB, Hkv, bs, D, dtype=torch.float16, device=cuda_device)
    vc = torch.zeros_like(kc)
    rk, rv = bits(kc).copy(), bits(vc).copy()
    cached_counts = []
    for sid, toks in enumerate(prompts):
        cached = bm.add_sequence_cached(sid, toks)
        assert cached == ref.add_sequence_cached(sid, toks)
        cached_counts.append(cached)
        t, _ = bm.tables([sid])
        assert list(t[0][: len(ref.tables[sid])]) == ref.tables[sid]
        # write K/V only for the tokens that are not already in the pool
        pos = np.arange(cached, len(toks))
        if len(pos) == 0:
            continue
        kv = np.stack([_kv_for_prefix(toks, int(p), Hkv, D) for p in pos])  # [n, 2, Hkv, D]
        k_new = torch.from_numpy(kv[:, 0]).half()
        v_new = torch.from_numpy(kv[:, 1]).half()
        slots = np.array([oracle.slot_of(ref.tables[sid], int(p), bs) for p in pos], np.int64)
        pkv.paged_kv_append(k_new.to(cuda_device), v_new.to(cuda_device), torch.from_numpy(slots).to(cuda_device),
                            kc, vc)
        oracle.append(bits(k_new), bits(v_new), oracle.F16, slots, rk, rv, oracle.F16)
    assert cached_counts == [0, 48, 48, 48, 0]
    t_first, _ = bm.tables([0])
    for sid in (1, 2, 3):
        t, _ = bm.tables([sid])
        assert list(t[0][:3]) == list(t_first[0][:3])  # the system prompt's full blocks are shared
    ids = np.arange(len(prompts))
    tables, lens = bm.tables(ids)
    q = torch.randn(len(prompts), Hq, D, generator=torch.Generator().manual_seed(5)).half()
    out = pkv.paged_attention_decode(q.to(cuda_device), kc, vc, torch.from_numpy(tables).to(cuda_device),
                                     torch.from_numpy(lens).to(cuda_device), 0.125)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    want = oracle.paged_decode(bits(q), oracle.F16, rk, rv, oracle.F16, tables, lens, 0.125)
    assert_attention_close(out, want, TOL["f16"])
    # and each request's attention equals attention over its own, unshared K/V
    for sid, toks in enumerate(prompts):
        kv = np.stack([_kv_for_prefix(toks, p, Hkv, D) for p in range(len(toks))])
        K = torch.from_numpy(kv[:, 0]).half().double().permute(1, 0, 2)  # [Hkv, L, D]
        V = torch.from_numpy(kv[:, 1]).half().double().permute(1, 0, 2)
        qq = q[sid].double().view(Hkv, Hq // Hkv, 1, D)
        o = torch.nn.functional.scaled_dot_product_attention(qq, K[:, None].expand(Hkv, Hq // Hkv, -1, D),
                                                             V[:, None].expand(Hkv, Hq // Hkv, -1, D), scale=0.125)
        assert np.abs(o.reshape(Hq, D).numpy() - want[sid]).max() < 1e-9
    assert pkv.device_error(reset=True) == 0


@pytest.mark.parametrize("act,Hq,Hkv,D", [("f16", 8, 8, 64), ("bf16", 32, 8, 128)])
def test_second_turn_reuses_answer_blocks_decode_matches_oracle(pkv_lib, cuda_device, act, Hq, Hkv, D):
    """A two-turn dialogue on the GPU.  Turn 1 writes its prompt's K/V, then
    decodes its answer token by token (the fused append + decode launch, slots
    from append_tokens, so the blocks the answer fills are registered).  Turn
    2's prompt is turn 1's prompt + answer + a new user turn: every full block
    of turn 1 is reused, only the rest is written, and the decode over the
    shared blocks matches the float64 oracle on the oracle allocator's tables
    and caches, and attention over the request's own unshared K/V."""
    pkv = pkv_lib
    pkv.device_error(reset=True)
    dt = torch.float16 if act == "f16" else torch.bfloat16
    code = oracle.F16 if act == "f16" else oracle.BF16
    bs, NB, scale = 16, 96, 1.0 / np.sqrt(D)
    rng = np.random.default_rng(11)
    prompt = list(rng.integers(0, 30000, size=77))
    answer = list(rng.integers(0, 30000, size=58))  # prompt + answer = 135 tokens: 8 full blocks
    user = list(rng.integers(0, 30000, size=21))
    bm = pkv.BlockManager(NB, bs)
    ref = RefBlockManager(NB, bs)
    kc = torch.zeros(NB, Hkv, bs, D, dtype=dt, device=cuda_device)
    vc = torch.zeros_like(kc)
    rk, rv = bits(kc).copy(), bits(vc).copy()
    gq = torch.Generator().manual_seed(7)

    def kv_rows(toks, positions):
        kv = np.stack([_kv_for_prefix(toks, int(p), Hkv, D) for p in positions])
        return torch.from_numpy(kv[:, 0]).to(dt), torch.from_numpy(kv[:, 1]).to(dt)

    def write_prompt(sid, toks):
        cached = bm.add_sequence_cached(sid, toks)
        assert cached == ref.add_sequence_cached(sid, toks)
        pos = np.arange(cached, len(toks))
        k_new, v_new = kv_rows(toks, pos)
        slots = np.array([oracle.slot_of(ref.tables[sid], int(p), bs) for p in pos], np.int64)
        pkv.paged_kv_append(k_new.to(cuda_device), v_new.to(cuda_device), torch.from_numpy(slots).to(cuda_device),
                            kc, vc)
        oracle.append(bits(k_new), bits(v_new), code, slots, rk, rv, code)
        return cached

    assert write_prompt(0, prompt) == 0
    # turn 1's answer: each step appends the newest token (its id known) and decodes
    for i, tok in enumerate(answer):
        toks = prompt + answer[: i + 1]
        slots, pairs = bm.append_tokens([0], [tok])
        want_slot, want_pair = ref.append_token(0, tok)
        assert slots[0] == want_slot and len(pairs) == 0 and want_pair is None
        k_new, v_new = kv_rows(toks, [len(toks) - 1])
        tables, lens = bm.tables([0])
        q = torch.randn(1, Hq, D, generator=gq).to(dt)
        out = pkv.paged_attention_decode_append(q.to(cuda_device), k_new.to(cuda_device), v_new.to(cuda_device),
                                                torch.from_numpy(slots).to(cuda_device), kc, vc,
                                                torch.from_numpy(tables).to(cuda_device),
                                                torch.from_numpy(lens).to(cuda_device), scale)
        oracle.append(bits(k_new), bits(v_new), code, slots, rk, rv, code)
        if i in (0, len(answer) - 1):
            torch.cuda.synchronize()
            want = oracle.paged_decode(bits(q), code, rk, rv, code, tables, lens, scale)
            assert_attention_close(out, want, TOL[act])
    n1 = len(prompt) + len(answer)
    assert bm.num_cached_blocks == n1 // bs == len(ref.block_of_prefix)
    t1, _ = bm.tables([0])
    bm.free_sequence(0)
    ref.free_sequence(0)
    second = prompt + answer + user
    assert write_prompt(1, second) == (n1 // bs) * bs
    t2, lens2 = bm.tables([1])
    assert list(t2[0][: n1 // bs]) == list(t1[0][: n1 // bs])  # prompt and answer blocks reused
    q = torch.randn(1, Hq, D, generator=gq).to(dt)
    out = pkv.paged_attention_decode(q.to(cuda_device), kc, vc, torch.from_numpy(t2).to(cuda_device),
                                     torch.from_numpy(lens2).to(cuda_device), scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    want = oracle.paged_decode(bits(q), code, rk, rv, code, np.asarray([ref.tables[1]], np.int32), lens2, scale)
    assert_attention_close(out, want, TOL[act])
    # the shared blocks hold exactly the K/V turn 2 would have written itself
    kv = np.stack([_kv_for_prefix(second, p, Hkv, D) for p in range(len(second))])
    K = torch.from_numpy(kv[:, 0]).to(dt).double().permute(1, 0, 2)
    V = torch.from_numpy(kv[:, 1]).to(dt).double().permute(1, 0, 2)
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(q[0].double().view(Hkv, G, 1, D),
                                                         K[:, None].expand(Hkv, G, -1, D),
                                                         V[:, None].expand(Hkv, G, -1, D), scale=scale)
    assert np.abs(o.reshape(Hq, D).numpy() - want[0]).max() < 1e-9
    assert pkv.device_error(reset=True) == 0
