"""QUEST on the GPU: block min/max metadata (full and incremental) exact
against the oracle; top-K selection equal to the oracle's where the bounds
have a margin at the cut and a valid top-K everywhere; the whole step
(metadata, selection, sparse decode) within tolerance of the oracle's own
selection followed by the oracle's sparse decode, on every (sequence, kv
head) whose cut has a margin; a budget covering every block reproduces full
decode."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager_ref import RefBlockManager
from tests.parity import ACT_CODE, TOL, assert_attention_close, bits

pytestmark = pytest.mark.gpu
DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture
def pkv(pkv_lib, cuda_device):
    pkv_lib.device_error(reset=True)
    prev = pkv_lib.set_kernel_path(pkv_lib.PATH_AUTO)
    yield pkv_lib
    pkv_lib.set_kernel_path(prev)
    assert pkv_lib.device_error(reset=True) == 0


def _setup(act, Hq, Hkv, D, bs, ctx, seed):
    g = torch.Generator().manual_seed(seed)
    B = len(ctx)
    NB = sum(-(-(c + 1) // bs) for c in ctx) + 3
    ref = RefBlockManager(NB, bs, free_list=torch.randperm(NB, generator=g).numpy())
    for i, c in enumerate(ctx):
        ref.add_sequence(i, c)
    slots = np.array([ref.append_slot(i)[0] for i in range(B)], np.int64)
    maxb = max(len(t) for t in ref.tables.values())
    tables = np.zeros((B, maxb), np.int32)
    for i in range(B):
        tables[i, : len(ref.tables[i])] = ref.tables[i]
    kc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
    vc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
    q = torch.randn(B, Hq, D, generator=g).to(DT[act])
    k_new = torch.randn(B, Hkv, D, generator=g).to(DT[act])
    v_new = torch.randn(B, Hkv, D, generator=g).to(DT[act])
    return q, kc, vc, k_new, v_new, tables, slots, np.array([c + 1 for c in ctx], np.int32)


CASES = [("bf16", 8, 8, 128, 16), ("f16", 16, 4, 64, 32), ("bf16", 32, 4, 128, 16), ("bf16", 16, 8, 64, 16),
         ("f16", 32, 4, 64, 16)]


MARGIN = 1e-4  # relative gap between the K-th and (K+1)-th oracle bounds that fixes the selection


def _check_selection(sel_h, slen_h, q, kbits, act, tables, lens, bs, budget):
    """Selected blocks equal the oracle's where its bounds have a margin at the
    cut, and form a valid top-K (ascending, distinct, token count right)
    everywhere.  Returns the oracle's selection (tables, lengths) and a
    [B, Hkv] mask of the rows whose selection is unique (a margin at the cut,
    or every block kept)."""
    want_sel, want_len, bounds = oracle.quest_select(bits(q), ACT_CODE[DT[act]], kbits, ACT_CODE[DT[act]],
                                                     tables, lens, budget)
    B, Hkv = slen_h.shape
    unique = np.zeros((B, Hkv), bool)
    for b in range(B):
        n = -(-int(lens[b]) // bs)
        pos = {int(x): j for j, x in enumerate(tables[b, :n])}
        for h in range(Hkv):
            got = [int(x) for x in sel_h[b, h, : min(budget, n)]]
            logical = [pos[x] for x in got]
            assert logical == sorted(logical) and len(set(logical)) == len(logical)
            toks = sum(int(lens[b]) - j * bs if j == n - 1 else bs for j in logical)
            assert slen_h[b, h] == toks
            if n <= budget:
                assert logical == list(range(n))
                unique[b, h] = True
                continue
            u = bounds[b, h, :n]
            order = np.sort(u)[::-1]
            cut, nxt = order[budget - 1], order[budget]
            # the kernel's float32 bounds are sums of 2 x head_dim non-negative
            # products (exact), so their relative error is below 256 * 2^-24 =
            # 1.5e-5; a gap of 1e-4 at the cut decides the selection
            if cut - nxt > MARGIN * max(1.0, abs(cut)):
                assert got == [int(x) for x in want_sel[b, h, :budget]]
                unique[b, h] = True
            else:  # a near tie at the cut: any valid top-K
                assert min(u[logical]) >= nxt - MARGIN * max(1.0, abs(nxt))
    return want_sel, want_len, unique


def _assert_rows_close(out, want, unique, group, tol):
    """Compare the output heads of the (sequence, kv head) rows marked unique."""
    B, Hkv = unique.shape
    rows = [(b, h * group + g) for b in range(B) for h in range(Hkv) if unique[b, h] for g in range(group)]
    assert len(rows) >= 0.75 * B * Hkv * group, "too few rows with a unique selection to compare"
    bi = torch.tensor([r[0] for r in rows])
    hi = torch.tensor([r[1] for r in rows])
    assert_attention_close(out.cpu()[bi, hi], want[bi.numpy(), hi.numpy()], tol)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_quest_metadata_selection_and_sparse_decode(pkv, case):
    act, Hq, Hkv, D, bs = case
    ctx = [0, 9, 100, 511, 1500, 3000]
    q, kc, vc, k_new, v_new, tables, slots, lens = _setup(act, Hq, Hkv, D, bs, ctx, zlib.crc32(repr(case).encode()))
    dev = torch.device("cuda")
    dk, dv = kc.to(dev), vc.to(dev)
    t_d, l_d = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
    # metadata of the cache before the step, then widened by the step's appended keys
    l0 = torch.from_numpy(np.maximum(lens - 1, 1)).to(dev)
    kmeta = pkv.quest_block_minmax(dk, t_d, l0)
    has_prev = lens > 1  # sequence 0 had no tokens before this step
    pkv.paged_kv_append(k_new.to(dev), v_new.to(dev), torch.from_numpy(slots).to(dev), dk, dv)
    pkv.quest_append_minmax(k_new.to(dev), torch.from_numpy(slots).to(dev), kmeta, bs)
    full = pkv.quest_block_minmax(dk, t_d, l_d)
    torch.cuda.synchronize()
    kbits = bits(dk)
    mn, mx = oracle.quest_block_minmax(kbits, ACT_CODE[DT[act]], tables, lens)
    meta = kmeta.float().cpu().numpy().astype(np.float64)
    meta_full = full.float().cpu().numpy().astype(np.float64)
    for b in range(len(ctx)):
        for j in range(-(-int(lens[b]) // bs)):
            blk = tables[b, j]
            np.testing.assert_array_equal(meta_full[blk, :, 0], mn[b, j])
            np.testing.assert_array_equal(meta_full[blk, :, 1], mx[b, j])
            if has_prev[b] or j > 0:
                np.testing.assert_array_equal(meta[blk], meta_full[blk])  # incremental == recompute
    for budget in (1, 8, 40):
        # the whole step on the GPU: metadata -> selection -> sparse decode
        sel, slen = pkv.quest_select(q.to(dev), full, t_d, l_d, bs, budget)
        out = pkv.paged_attention_decode_sparse(q.to(dev), dk, dv, sel, slen, 0.09)
        torch.cuda.synchronize()
        want_sel, want_len, unique = _check_selection(sel.cpu().numpy(), slen.cpu().numpy(), q, kbits, act, tables,
                                                      lens, bs, budget)
        # the oracle's own selection, then the oracle's sparse decode
        want = oracle.sparse_decode(bits(q), ACT_CODE[DT[act]], kbits, bits(dv), ACT_CODE[DT[act]], want_sel,
                                    want_len, 0.09)
        _assert_rows_close(out, want, unique, Hq // Hkv, TOL[act])


def test_full_budget_reproduces_full_decode(pkv):
    q, kc, vc, _, _, tables, _, lens = _setup("bf16", 8, 8, 128, 16, [50, 700, 2000], 3)
    dev = torch.device("cuda")
    dk, dv = kc.to(dev), vc.to(dev)
    t_d, l_d = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
    kmeta = pkv.quest_block_minmax(dk, t_d, l_d)
    sel, slen = pkv.quest_select(q.to(dev), kmeta, t_d, l_d, 16, tables.shape[1])
    sparse = pkv.paged_attention_decode_sparse(q.to(dev), dk, dv, sel, slen, 0.09)
    full = pkv.paged_attention_decode(q.to(dev), dk, dv, t_d, l_d, 0.09)
    torch.cuda.synchronize()
    assert torch.equal(sparse, full)


@pytest.mark.parametrize("path", [1, 3])
def test_sparse_decode_paths_agree_with_oracle(pkv, path):
    """Per-(sequence, kv head) tables on the CUDA-core and tensor-core kernels."""
    q, kc, vc, _, _, tables, _, lens = _setup("bf16", 32, 4, 128, 16, [100, 900, 2500, 4000], 21)
    dev = torch.device("cuda")
    dk, dv = kc.to(dev), vc.to(dev)
    t_d, l_d = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
    kmeta = pkv.quest_block_minmax(dk, t_d, l_d)
    sel, slen = pkv.quest_select(q.to(dev), kmeta, t_d, l_d, 16, 64)
    pkv.set_kernel_path(path)
    out = pkv.paged_attention_decode_sparse(q.to(dev), dk, dv, sel, slen, 0.088, partition_size=512)
    torch.cuda.synchronize()
    want_sel, want_len, unique = _check_selection(sel.cpu().numpy(), slen.cpu().numpy(), q, bits(kc), "bf16",
                                                  tables, lens, 16, 64)
    want = oracle.sparse_decode(bits(q), oracle.BF16, bits(dk), bits(dv), oracle.BF16, want_sel, want_len, 0.088)
    _assert_rows_close(out, want, unique, 32 // 4, TOL["bf16"])


@pytest.mark.parametrize("Hkv,group,D", [(2, 4, 64), (2, 8, 64), (8, 4, 128), (16, 8, 128), (8, 1, 64)])
def test_quest_select_many_items_per_cta(pkv, Hkv, group, D):
    """Enough (sequence, kv-head group, chunk) items that every persistent CTA
    of the bounds kernel cycles its shared-memory ring several times and, with
    8 or more kv heads (groups of 8 loaded by TMA boxes), rewrites its query
    operand for several (sequence, group) pairs."""
    bs = 16
    ctx = [18000 // Hkv + 37 * i for i in range(96)]  # 96 sequences x (9 to 23 chunks) per group
    q, kc, _, _, _, tables, _, lens = _setup("bf16", Hkv * group, Hkv, D, bs, ctx, 77 + group + Hkv)
    dev = torch.device("cuda")
    dk = kc.to(dev)
    t_d, l_d = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
    kmeta = pkv.quest_block_minmax(dk, t_d, l_d)
    for budget in (3, 100):
        sel, slen = pkv.quest_select(q.to(dev), kmeta, t_d, l_d, bs, budget)
        torch.cuda.synchronize()
        _check_selection(sel.cpu().numpy(), slen.cpu().numpy(), q, bits(kc), "bf16", tables, lens, bs, budget)


@pytest.mark.parametrize("path", [1, 3])
def test_sparse_decode_e4m3_cache(pkv, path):
    """Per-(sequence, kv head) block lists over an E4M3 cache (chosen here, in
    random order, with the partly filled last block at the end of some
    lists), on the CUDA-core and tensor-core kernels."""
    g = torch.Generator().manual_seed(96)
    rng = np.random.default_rng(96)
    B, Hq, Hkv, D, bs = 5, 32, 4, 128, 16
    lens = [37, 400, 1000, 1537, 2048]
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + 4
    perm = torch.randperm(NB, generator=g).numpy()
    owned, o = [], 0
    for n in nblk:
        owned.append(perm[o:o + n])
        o += n
    maxsel = max(nblk)
    sel = np.zeros((B, Hkv, maxsel), np.int32)
    slen = np.zeros((B, Hkv), np.int32)
    for b, L in enumerate(lens):
        full, tail = L // bs, L % bs
        for h in range(Hkv):
            k = int(rng.integers(1, full + 1)) if full else 0
            picks = list(rng.permutation(owned[b][:full])[:k])
            n_tok = k * bs
            if tail and (rng.random() < 0.5 or k == 0):
                picks.append(owned[b][full])  # the partly filled block, last
                n_tok += tail
            sel[b, h, :len(picks)] = picks
            slen[b, h] = n_tok
    kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
    vc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
    kc[(kc & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x3C
    q = torch.randn(B, Hq, D, generator=g).bfloat16()
    ks, vs, scale = 0.021, 0.013, 0.088
    dev = torch.device("cuda")
    pkv.set_kernel_path(path)
    out = pkv.paged_attention_decode_sparse(q.to(dev), kc.to(dev), vc.to(dev), torch.from_numpy(sel).to(dev),
                                            torch.from_numpy(slen).to(dev), scale,
                                            k_scale=torch.tensor([ks], device=dev),
                                            v_scale=torch.tensor([vs], device=dev))
    torch.cuda.synchronize()
    want = oracle.sparse_decode(bits(q), oracle.BF16, kc.numpy(), vc.numpy(), oracle.E4M3, sel, slen, scale,
                                k_scale=ks, v_scale=vs)
    assert_attention_close(out, want, TOL["e4m3"])


@pytest.mark.parametrize("act,Hq,Hkv,D,bs", [("bf16", 32, 4, 128, 16), ("f16", 16, 8, 64, 32)])
def test_quest_e4m3_cache_metadata_selection_and_step(pkv, act, Hq, Hkv, D, bs):
    """QUEST over an E4M3 cache: metadata (full, and widened by a step's keys
    that the append quantises with k_scale) equal to the oracle's decoded
    codes; selection equal to the oracle's (which scales the bounds by
    k_scale) where the cut has a margin; the whole step's output within the
    E4M3 tolerance of the oracle's sparse decode on its own selection."""
    g = torch.Generator().manual_seed(Hq + D)
    ctx = [0, 40, 700, 2000, 2900]
    B = len(ctx)
    NB = sum(-(-(c + 1) // bs) for c in ctx) + 3
    ref = RefBlockManager(NB, bs, free_list=torch.randperm(NB, generator=g).numpy())
    for i, c in enumerate(ctx):
        ref.add_sequence(i, c)
    slots = np.array([ref.append_slot(i)[0] for i in range(B)], np.int64)
    maxb = max(len(t) for t in ref.tables.values())
    tables = np.zeros((B, maxb), np.int32)
    for i in range(B):
        tables[i, : len(ref.tables[i])] = ref.tables[i]
    lens = np.array([c + 1 for c in ctx], np.int32)
    kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
    vc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
    kc[(kc & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x3C
    q = torch.randn(B, Hq, D, generator=g).to(DT[act])
    k_new = torch.randn(B, Hkv, D, generator=g).to(DT[act])
    v_new = torch.randn(B, Hkv, D, generator=g).to(DT[act])
    ks, vs = 0.0123, 0.0171
    dev = torch.device("cuda")
    dk, dv = kc.to(dev), vc.to(dev)
    ksd, vsd = torch.tensor([ks], device=dev), torch.tensor([vs], device=dev)
    t_d, l_d = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
    l0 = torch.from_numpy(np.maximum(lens - 1, 1)).to(dev)
    kmeta = pkv.quest_block_minmax(dk, t_d, l0, meta_dtype=DT[act])
    pkv.paged_kv_append(k_new.to(dev), v_new.to(dev), torch.from_numpy(slots).to(dev), dk, dv, ksd, vsd)
    pkv.quest_append_minmax(k_new.to(dev), torch.from_numpy(slots).to(dev), kmeta, bs, k_scale=ksd)
    full = pkv.quest_block_minmax(dk, t_d, l_d, meta_dtype=DT[act])
    torch.cuda.synchronize()
    kbits = dk.cpu().numpy()
    # the appended codes are the oracle's
    rk, rv = kc.numpy().copy(), vc.numpy().copy()
    oracle.append(bits(k_new), bits(v_new), ACT_CODE[DT[act]], slots, rk, rv, oracle.E4M3, k_scale=ks, v_scale=vs)
    assert np.array_equal(kbits, rk) and np.array_equal(dv.cpu().numpy(), rv)
    mn, mx = oracle.quest_block_minmax(kbits, oracle.E4M3, tables, lens)
    meta = kmeta.float().cpu().numpy().astype(np.float64)
    meta_full = full.float().cpu().numpy().astype(np.float64)
    for b in range(B):
        for j in range(-(-int(lens[b]) // bs)):
            blk = tables[b, j]
            np.testing.assert_array_equal(meta_full[blk, :, 0], mn[b, j])
            np.testing.assert_array_equal(meta_full[blk, :, 1], mx[b, j])
            if lens[b] > 1 or j > 0:
                np.testing.assert_array_equal(meta[blk], meta_full[blk])  # incremental == recompute
    for budget in (2, 16):
        sel, slen = pkv.quest_select(q.to(dev), full, t_d, l_d, bs, budget)
        out = pkv.paged_attention_decode_sparse(q.to(dev), dk, dv, sel, slen, 0.08, k_scale=ksd, v_scale=vsd)
        torch.cuda.synchronize()
        want_sel, want_len, bounds = oracle.quest_select(bits(q), ACT_CODE[DT[act]], kbits, oracle.E4M3, tables,
                                                         lens, budget, k_scale=ks)
        sel_h, slen_h = sel.cpu().numpy(), slen.cpu().numpy()
        unique = np.zeros((B, Hkv), bool)
        for b in range(B):
            n = -(-int(lens[b]) // bs)
            for h in range(Hkv):
                if n <= budget:
                    unique[b, h] = True
                    assert list(sel_h[b, h, :n]) == list(tables[b, :n]) and slen_h[b, h] == lens[b]
                    continue
                order = np.sort(bounds[b, h, :n])[::-1]
                if order[budget - 1] - order[budget] > MARGIN * max(1.0, abs(order[budget - 1])):
                    unique[b, h] = True
                    assert list(sel_h[b, h, :budget]) == list(want_sel[b, h, :budget])
                    assert slen_h[b, h] == want_len[b, h]
        want = oracle.sparse_decode(bits(q), ACT_CODE[DT[act]], kbits, dv.cpu().numpy(), oracle.E4M3, want_sel,
                                    want_len, 0.08, k_scale=ks, v_scale=vs)
        _assert_rows_close(out, want, unique, Hq // Hkv, TOL["e4m3"])
