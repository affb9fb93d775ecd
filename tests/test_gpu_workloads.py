"""Full-size decode steps of each workload, in the launch configuration the
benchmark times (the append fused into the decode launch, library-chosen
partition size and kernel path), checked against the float64 oracle on every
sequence of the batch: the block manager's tables and slots against the
oracle allocator, the append bit for bit on every block the batch uses, and
every attention output element within the tolerance."""
import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager_ref import RefBlockManager
from paged_kv_cache_102_gb300 import workloads as W
from tests.parity import ACT_CODE, TOL, assert_attention_close, bits, compact_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv(pkv_lib, cuda_device):
    pkv_lib.device_error(reset=True)
    yield pkv_lib
    assert pkv_lib.device_error(reset=True) == 0, "a kernel flagged a device-side error"


def _cache_code(wl):
    return oracle.E4M3 if wl.cache_dtype == "e4m3" else ACT_CODE[W.DTYPES[wl.cache_dtype]]




WORKLOADS = ["tiny", "llama7b", "gqa_bs16", "gqa_bs32", "fp8_13b", "long_gqa", "gqa_fp8", "gqa_g2", "gqa_d64"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_decode_step(pkv, name):
    d = W.draw(name, seed=0)
    wl = d.workload
    dev = torch.device("cuda")
    vals = W.make_values(d, device=dev)
    B = len(d.context_lens)
    ids = np.arange(B)
    bm = pkv.BlockManager(d.num_blocks, wl.block_size, free_list=d.free_list)
    ref = RefBlockManager(d.num_blocks, wl.block_size, free_list=d.free_list)
    for i, c in enumerate(d.context_lens):
        bm.add_sequence(i, int(c))
        ref.add_sequence(i, int(c))
    slots, pairs = bm.append_slots(ids)
    want_slots = [ref.append_slot(i) for i in ids]
    assert list(slots) == [s for s, _ in want_slots] and len(pairs) == 0
    tables, lens = bm.tables(ids)
    for i in ids:
        assert list(tables[i, : len(ref.tables[i])]) == ref.tables[i]
    assert np.array_equal(lens, d.context_lens + 1)

    pick = ids  # the whole batch
    kc0, vc0, t2 = compact_pool(vals["k_cache"], vals["v_cache"], tables[pick], lens[pick], wl.block_size)
    ks = vals.get("k_scale")
    vs = vals.get("v_scale")

    # device: the append fused into the decode launch, as the benchmark times it
    out = pkv.paged_attention_decode_append(vals["q"], vals["k_new"], vals["v_new"], torch.from_numpy(slots).to(dev),
                                            vals["k_cache"], vals["v_cache"], torch.from_numpy(tables).to(dev),
                                            torch.from_numpy(lens).to(dev), wl.scale, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()

    # oracle on every sequence, on the compacted copy of the blocks the batch uses
    rk, rv = bits(kc0).copy(), bits(vc0).copy()
    s2 = np.array([oracle.slot_of(t2[j], int(lens[i]) - 1, wl.block_size) for j, i in enumerate(pick)], np.int64)
    act = ACT_CODE[W.DTYPES[wl.act_dtype]]
    ksf = float(ks.item()) if ks is not None else 1.0
    vsf = float(vs.item()) if vs is not None else 1.0
    oracle.append(bits(vals["k_new"][pick]), bits(vals["v_new"][pick]), act, s2, rk, rv, _cache_code(wl),
                  k_scale=ksf, v_scale=vsf)
    kc1, vc1, _ = compact_pool(vals["k_cache"], vals["v_cache"], tables[pick], lens[pick], wl.block_size)
    assert np.array_equal(bits(kc1), rk) and np.array_equal(bits(vc1), rv), "append differs from the oracle"
    want = oracle.paged_decode(bits(vals["q"][pick]), act, rk, rv, _cache_code(wl), t2, lens[pick], wl.scale,
                               k_scale=ksf, v_scale=vsf)
    tol = TOL["e4m3"] if wl.cache_dtype == "e4m3" else TOL[wl.act_dtype]
    assert_attention_close(out, want, tol, label=name)


def test_shared_prefix_parallel_sampling(pkv):
    """32 prompts x 4 samples sharing the prompt's blocks (ref count 4); each
    sample appends its divergent tokens one step at a time (copy-on-write of
    the partial last block on the first divergent write), then one more token
    and a decode step.  The oracle replays the same steps with its own
    allocator, copy and append, and attends on every sequence."""
    d = W.draw("shared_prefix", seed=0)
    wl = d.workload
    dev = torch.device("cuda")
    vals = W.make_values(d, device=dev)
    n = wl.samples_per_prompt
    S = len(d.context_lens)
    bm = pkv.BlockManager(d.num_blocks, wl.block_size, free_list=d.free_list)
    ref = RefBlockManager(d.num_blocks, wl.block_size, free_list=d.free_list)
    for p, plen in enumerate(d.prompt_lens):
        bm.add_sequence(p * n, int(plen))
        ref.add_sequence(p * n, int(plen))
        for j in range(1, n):
            bm.fork(p * n, p * n + j)
            ref.fork(p * n, p * n + j)
    for b in ref.tables[0]:
        assert bm.ref_count(b) == ref.ref[b] == n
    rk, rv = bits(vals["k_cache"]).copy(), bits(vals["v_cache"]).copy()
    act = ACT_CODE[W.DTYPES[wl.act_dtype]]
    g = torch.Generator(device=dev)
    g.manual_seed(1000)
    max_div = int(d.divergent.max())
    total_pairs = 0
    for step in range(max_div + 1):
        if step < max_div:
            active = np.nonzero(d.divergent > step)[0]
        else:
            active = np.arange(S)  # the decode step's own token
        kn = torch.randn(len(active), wl.num_kv_heads, wl.head_dim, generator=g, device=dev).to(W.DTYPES[wl.act_dtype])
        vn = torch.randn(len(active), wl.num_kv_heads, wl.head_dim, generator=g, device=dev).to(W.DTYPES[wl.act_dtype])
        slots, pairs = bm.append_slots(active)
        want = [ref.append_slot(int(s)) for s in active]
        assert list(slots) == [w[0] for w in want]
        assert [tuple(p) for p in pairs] == [w[1] for w in want if w[1] is not None]
        total_pairs += len(pairs)
        if len(pairs):
            pkv.paged_block_copy(vals["k_cache"], vals["v_cache"], torch.from_numpy(pairs).to(dev))
            oracle.block_copy(rk, rv, pairs)
        pkv.paged_kv_append(kn, vn, torch.from_numpy(slots).to(dev), vals["k_cache"], vals["v_cache"])
        oracle.append(bits(kn), bits(vn), act, slots, rk, rv, act)
    # every prompt's partial last block was copied by 3 of its 4 samples (the last holder writes in place)
    assert total_pairs == (n - 1) * wl.batch
    ids = np.arange(S)
    tables, lens = bm.tables(ids)
    assert np.array_equal(lens, d.context_lens + 1)
    out = pkv.paged_attention_decode(vals["q"], vals["k_cache"], vals["v_cache"], torch.from_numpy(tables).to(dev),
                                     torch.from_numpy(lens).to(dev), wl.scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(vals["k_cache"]), rk) and np.array_equal(bits(vals["v_cache"]), rv)
    want = oracle.paged_decode(bits(vals["q"]), act, rk, rv, act, tables, lens, wl.scale)
    assert_attention_close(out, want, TOL[wl.act_dtype], label="shared_prefix")
    # memory side of parallel sampling: shared prompt blocks are stored once
    unique = len({b for s in ids for b in ref.tables[int(s)]})
    logical = sum(len(ref.tables[int(s)]) for s in ids)
    assert unique < logical
