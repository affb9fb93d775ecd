"""GPU parity of the three kernels against the float64 oracle, through the
C ABI (via the thin binding).  Append and block copy must be bit-exact;
attention must be within the stated tolerance of the float64 oracle."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager_ref import RefBlockManager
from tests.parity import ACT_CODE, TOL, assert_attention_close, bits

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def pkv(pkv_lib, cuda_device):
    pkv_lib.device_error(reset=True)
    yield pkv_lib
    assert pkv_lib.device_error(reset=True) == 0, "a kernel flagged a device-side error"


def _gen(seed):
    return torch.Generator().manual_seed(seed)


# ----------------------------------------------------------------- append ---
@pytest.mark.parametrize("act,cache,Hkv,D,bs,T", [
    ("f16", "f16", 8, 64, 16, 4),
    ("bf16", "bf16", 32, 128, 16, 64),
    ("bf16", "bf16", 8, 128, 32, 300),
    ("f16", "f16", 3, 40, 5, 17),
    ("bf16", "e4m3", 40, 128, 16, 256),
    ("f16", "e4m3", 8, 64, 32, 33),
])
def test_append_bit_exact(pkv, act, cache, Hkv, D, bs, T):
    g = _gen(T * 7 + D)
    NB = T // bs + 8
    k = (torch.randn(T, Hkv, D, generator=g) * 3).to(DT[act])
    v = (torch.randn(T, Hkv, D, generator=g) * 3).to(DT[act])
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[::5] = -1  # padding tokens are skipped
    if cache == "e4m3":
        kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
        ks, vs = torch.tensor([0.011], dtype=torch.float32), torch.tensor([0.027], dtype=torch.float32)
    else:
        kc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
        ks = vs = None
    vc = kc.clone()
    ref_k, ref_v = bits(kc).copy(), bits(vc).copy()
    code = oracle.E4M3 if cache == "e4m3" else ACT_CODE[DT[act]]
    oracle.append(bits(k), bits(v), ACT_CODE[DT[act]], slots.numpy(), ref_k, ref_v, code,
                  k_scale=1.0 if ks is None else float(ks), v_scale=1.0 if vs is None else float(vs))
    dk, dv = kc.cuda(), vc.cuda()
    pkv.paged_kv_append(k.cuda(), v.cuda(), slots.cuda(), dk, dv,
                        None if ks is None else ks.cuda(), None if vs is None else vs.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(dk), ref_k)
    assert np.array_equal(bits(dv), ref_v)


def test_append_e4m3_rounding_sweep(pkv):
    """Every E4M3 decision (ties, subnormals, saturation) matches the oracle's encoder."""
    g = _gen(99)
    Hkv, D, bs = 1, 128, 16
    T = 4096
    x = torch.cat([torch.randn(T * D // 2, generator=g) * 200, torch.randn(T * D // 2, generator=g) * 0.02])
    mids = torch.from_numpy(oracle.decode_elements(np.arange(0, 0x7F, dtype=np.uint8), oracle.E4M3))
    mids = ((mids[:-1] + mids[1:]) / 2).float()
    x[: mids.numel()] = mids
    x[mids.numel(): 2 * mids.numel()] = -mids
    k = x.reshape(T, Hkv, D).to(torch.bfloat16)
    slots = torch.arange(T, dtype=torch.int64)
    kc = torch.zeros(T // bs, Hkv, bs, D, dtype=torch.uint8)
    ref_k, ref_v = bits(kc).copy(), bits(kc).copy()
    oracle.append(bits(k), bits(k), oracle.BF16, slots.numpy(), ref_k, ref_v, oracle.E4M3, k_scale=1.0, v_scale=0.5)
    dk, dv = kc.cuda(), kc.clone().cuda()
    one = torch.tensor([1.0], device="cuda")
    half = torch.tensor([0.5], device="cuda")
    pkv.paged_kv_append(k.cuda(), k.cuda(), slots.cuda(), dk, dv, one, half)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dk), ref_k) and np.array_equal(bits(dv), ref_v)


def test_append_flags_bad_slot(pkv):
    NB, Hkv, bs, D = 4, 2, 16, 64
    k = torch.randn(2, Hkv, D, dtype=torch.float16, device="cuda")
    kc = torch.zeros(NB, Hkv, bs, D, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([NB * bs, 3], dtype=torch.int64, device="cuda")
    pkv.paged_kv_append(k, k, slots, kc, vc)
    assert pkv.device_error(reset=True) == pkv.DEV_BAD_SLOT
    assert torch.equal(kc[0, :, 3], k[1])  # the valid token still landed
    assert kc.count_nonzero() == k[1].count_nonzero()


# ------------------------------------------------------------- block copy ---
@pytest.mark.parametrize("Hkv,bs,D,dtype,P", [(32, 16, 128, torch.float16, 7), (8, 32, 64, torch.bfloat16, 33),
                                              (40, 16, 128, torch.uint8, 5), (1, 4, 8, torch.float16, 3)])
def test_block_copy_bit_exact(pkv, Hkv, bs, D, dtype, P):
    g = _gen(P)
    NB = 3 * P + 4
    if dtype == torch.uint8:
        kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=dtype, generator=g)
        vc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=dtype, generator=g)
    else:
        kc = torch.randn(NB, Hkv, bs, D, generator=g).to(dtype)
        vc = torch.randn(NB, Hkv, bs, D, generator=g).to(dtype)
    perm = torch.randperm(NB, generator=g)
    pairs = torch.stack([perm[:P], perm[P:2 * P]], dim=1).to(torch.int32).contiguous()
    rk, rv = bits(kc).copy(), bits(vc).copy()
    oracle.block_copy(rk, rv, pairs.numpy())
    dk, dv = kc.cuda(), vc.cuda()
    pkv.paged_block_copy(dk, dv, pairs.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(dk), rk) and np.array_equal(bits(dv), rv)


def test_block_copy_flags_bad_pair(pkv):
    kc = torch.randn(4, 2, 16, 64, device="cuda").half()
    vc = kc.clone()
    before = kc.clone()
    pairs = torch.tensor([[0, 4], [1, 2]], dtype=torch.int32, device="cuda")
    pkv.paged_block_copy(kc, vc, pairs)
    assert pkv.device_error(reset=True) == pkv.DEV_BAD_PAIR
    assert torch.equal(kc[2], before[1]) and torch.equal(kc[0], before[0])


# ----------------------------------------------------------------- decode ---
def _random_paged(g, B, Hq, Hkv, D, bs, lens, act, cache, extra_blocks=5):
    """Random pool, shuffled tables from the oracle allocator, queries."""
    nblk = [-(-int(L) // bs) for L in lens]
    NB = sum(nblk) + extra_blocks
    fl = torch.randperm(NB, generator=g).numpy().astype(np.int32)
    ref = RefBlockManager(NB, bs, free_list=fl)
    for i, L in enumerate(lens):
        ref.add_sequence(i, int(L))
    maxb = max(nblk) + 1
    tables = np.full((B, maxb), -7, np.int32)  # entries past a sequence's blocks are never read
    for i in range(B):
        tables[i, : nblk[i]] = ref.tables[i]
    q = torch.randn(B, Hq, D, generator=g).to(DT[act])
    if cache == "e4m3":
        kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
        vc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
        kc[(kc & 0x7F) == 0x7F] = 0x3C  # no NaN codes in the pool
        vc[(vc & 0x7F) == 0x7F] = 0x3C
    else:
        kc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
        vc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
    return q, kc, vc, tables, np.asarray(lens, np.int32)


def _run_decode(pkv, q, kc, vc, tables, lens, scale, partition_size, ks=None, vs=None):
    out = pkv.paged_attention_decode(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(tables).cuda(),
                                     torch.from_numpy(lens).cuda(), scale,
                                     k_scale=None if ks is None else torch.tensor([ks], device="cuda"),
                                     v_scale=None if vs is None else torch.tensor([vs], device="cuda"),
                                     partition_size=partition_size)
    torch.cuda.synchronize()
    return out


CASES = [
    # act, cache, Hq, Hkv, D, bs
    ("f16", "f16", 8, 8, 64, 16),
    ("bf16", "bf16", 4, 4, 128, 16),
    ("bf16", "bf16", 16, 2, 128, 32),
    ("f16", "f16", 8, 4, 64, 32),
    ("bf16", "bf16", 8, 2, 64, 16),
    ("bf16", "e4m3", 4, 4, 128, 16),
    ("f16", "e4m3", 8, 1, 64, 32),
    ("bf16", "e4m3", 16, 4, 128, 32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("partition_size", [0, -1, 32, 64, 128])
def test_decode_parity_sweep(pkv, case, partition_size):
    act, cache, Hq, Hkv, D, bs = case
    if partition_size > 0 and partition_size % bs:
        pytest.skip("partition must be a multiple of the block size")
    g = _gen(zlib.crc32(repr((case, partition_size)).encode()))
    lens = [1, 2, bs - 1, bs, bs + 1, 31, 32, 33, 64, 95, 129, 300, 517]
    B = len(lens)
    q, kc, vc, tables, lens = _random_paged(g, B, Hq, Hkv, D, bs, lens, act, cache)
    scale = 1.0 / math.sqrt(D)
    ks, vs = (0.0173, 0.031) if cache == "e4m3" else (1.0, 1.0)
    code = oracle.E4M3 if cache == "e4m3" else ACT_CODE[DT[act]]
    want = oracle.paged_decode(bits(q), ACT_CODE[DT[act]], bits(kc), bits(vc), code, tables, lens, scale,
                               k_scale=ks, v_scale=vs)
    got = _run_decode(pkv, q, kc, vc, tables, lens, scale, partition_size,
                      *((ks, vs) if cache == "e4m3" else (None, None)))
    assert_attention_close(got, want, TOL[cache if cache == "e4m3" else act])


def test_decode_closed_forms(pkv):
    """L = 1 gives v_0 exactly; equal keys give the mean of V."""
    g = _gen(5)
    B, H, D, bs = 3, 4, 128, 16
    q, kc, vc, tables, _ = _random_paged(g, B, H, H, D, bs, [1, 1, 1], "bf16", "bf16")
    lens = np.array([1, 1, 1], np.int32)
    out = _run_decode(pkv, q, kc, vc, tables, lens, 0.1, -1)
    v0 = torch.stack([vc[tables[b, 0], :, 0] for b in range(B)])
    assert torch.equal(out.cpu(), v0)
    # equal keys across a 100-token sequence -> uniform weights
    q, kc, vc, tables, _ = _random_paged(g, 1, H, H, D, bs, [100], "f16", "f16")
    kc[:] = kc[0, :, 0:1, :]
    out = _run_decode(pkv, q, kc, vc, tables, np.array([100], np.int32), 0.3, 32)
    blocks = [int(b) for b in tables[0, :7]]
    vals = torch.cat([vc[b] for b in blocks], dim=1)[:, :100].double().mean(dim=1)
    assert (out[0].cpu().double() - vals).abs().max() < 2e-3


def test_decode_long_context_split(pkv):
    """A 20000-token context, several partition sizes, vs the oracle."""
    g = _gen(11)
    q, kc, vc, tables, lens = _random_paged(g, 2, 8, 2, 128, 16, [20000, 12345], "bf16", "bf16")
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), oracle.BF16, tables, lens, 1 / math.sqrt(128))
    for ps in (0, 512, 2048):
        got = _run_decode(pkv, q, kc, vc, tables, lens, 1 / math.sqrt(128), ps)
        assert_attention_close(got, want, TOL["bf16"])


def test_decode_flags_bad_inputs(pkv):
    g = _gen(3)
    q, kc, vc, tables, lens = _random_paged(g, 2, 4, 4, 64, 16, [20, 40], "f16", "f16")
    bad_len = lens.copy()
    bad_len[1] = tables.shape[1] * 16 + 1
    _run_decode(pkv, q, kc, vc, tables, bad_len, 0.125, -1)
    assert pkv.device_error(reset=True) == pkv.DEV_BAD_CONTEXT_LEN
    bad_tab = tables.copy()
    bad_tab[0, 1] = kc.shape[0] + 3
    _run_decode(pkv, q, kc, vc, bad_tab, lens, 0.125, -1)
    assert pkv.device_error(reset=True) == pkv.DEV_BAD_BLOCK
    bad_len[1] = 0
    _run_decode(pkv, q, kc, vc, tables, bad_len, 0.125, 0)
    assert pkv.device_error(reset=True) == pkv.DEV_BAD_CONTEXT_LEN


def test_decode_empty_batch_and_streams(pkv):
    q = torch.empty(0, 4, 64, dtype=torch.float16, device="cuda")
    kc = torch.zeros(2, 4, 16, 64, dtype=torch.float16, device="cuda")
    out = pkv.paged_attention_decode(q, kc, kc, torch.zeros(0, 1, dtype=torch.int32, device="cuda"),
                                     torch.zeros(0, dtype=torch.int32, device="cuda"), 0.1)
    assert out.shape == (0, 4, 64)
    # a side stream is honoured
    g = _gen(8)
    q, kc, vc, tables, lens = _random_paged(g, 4, 8, 8, 64, 16, [40, 17, 33, 2], "f16", "f16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = pkv.paged_attention_decode(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(tables).cuda(),
                                         torch.from_numpy(lens).cuda(), 0.125, stream=s)
    s.synchronize()
    want = oracle.paged_decode(bits(q), oracle.F16, bits(kc), bits(vc), oracle.F16, tables, lens, 0.125)
    assert_attention_close(out, want, TOL["f16"])


# ------------------------------------------------------ tensor-core GQA path ---
TC_CASES = [
    # act, Hq, Hkv, bs, head_dim (64: pairs of kv heads per item)
    ("bf16", 16, 2, 16, 128),
    ("bf16", 32, 8, 32, 128),
    ("f16", 16, 4, 16, 128),
    ("bf16", 8, 4, 32, 128),
    ("f16", 8, 2, 16, 128),
    ("bf16", 64, 8, 16, 64),
    ("f16", 8, 2, 32, 64),
    ("bf16", 16, 4, 32, 64),
    ("f16", 8, 4, 16, 64),
]


@pytest.fixture
def kernel_path(pkv):
    prev = pkv.set_kernel_path(pkv.PATH_AUTO)
    yield pkv
    pkv.set_kernel_path(prev)


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("path", [2, 3])
@pytest.mark.parametrize("partition_size", [-1, 128, 256, 64])
def test_decode_tensor_core_parity(kernel_path, case, path, partition_size):
    pkv = kernel_path
    act, Hq, Hkv, bs, D = case
    if partition_size > 0 and partition_size % bs:
        pytest.skip("partition must be a multiple of the block size")
    if partition_size == -1 and Hq // Hkv < 4:
        partition_size = 512  # the library's own choice for group 2 is 1024, beyond the tensor-core kernel
    g = _gen(zlib.crc32(repr((case, path, partition_size)).encode()))
    lens = [1, 2, 15, 16, 17, 100, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1000, 1531]
    q, kc, vc, tables, lens = _random_paged(g, len(lens), Hq, Hkv, D, bs, lens, act, act)
    scale = 1.0 / math.sqrt(D)
    want = oracle.paged_decode(bits(q), ACT_CODE[DT[act]], bits(kc), bits(vc), ACT_CODE[DT[act]], tables, lens, scale)
    pkv.set_kernel_path(path)
    got = _run_decode(pkv, q, kc, vc, tables, lens, scale, partition_size)
    assert_attention_close(got, want, TOL[act])


TC_FP8_CASES = [
    # act, Hq, Hkv, bs (E4M3 cache)
    ("bf16", 32, 4, 16),
    ("f16", 16, 4, 32),
    ("bf16", 16, 8, 16),
]


@pytest.mark.parametrize("case", TC_FP8_CASES, ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("path", [2, 3])
@pytest.mark.parametrize("partition_size", [-1, 128, 256])
def test_decode_tensor_core_e4m3_parity(kernel_path, case, path, partition_size):
    """E4M3 cache on the tensor cores: E4M3 tiles straight into the MMA, q and
    P as E4M3 high + low parts, scales applied to S and O."""
    pkv = kernel_path
    act, Hq, Hkv, bs = case
    if partition_size > 0 and partition_size % bs:
        pytest.skip("partition must be a multiple of the block size")
    if partition_size == -1 and Hq // Hkv < 4:
        partition_size = 512
    g = _gen(zlib.crc32(repr(("e4m3", case, path, partition_size)).encode()))
    lens = [1, 2, 15, 16, 17, 100, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1000, 1531]
    q, kc, vc, tables, lens = _random_paged(g, len(lens), Hq, Hkv, 128, bs, lens, act, "e4m3")
    ks, vs, scale = 0.021, 0.013, 1.0 / math.sqrt(128)
    want = oracle.paged_decode(bits(q), ACT_CODE[DT[act]], bits(kc), bits(vc), oracle.E4M3, tables, lens, scale,
                               k_scale=ks, v_scale=vs)
    pkv.set_kernel_path(path)
    got = _run_decode(pkv, q, kc, vc, tables, lens, scale, partition_size, ks, vs)
    assert_attention_close(got, want, TOL["e4m3"])


def test_decode_tensor_core_e4m3_large_queries(kernel_path):
    """Queries far beyond the E4M3 range take the exact power-of-two pre-scale;
    a group whose queries are all zero gives the plain mean of V."""
    pkv = kernel_path
    g = _gen(91)
    lens = [40, 700, 1300]
    q, kc, vc, tables, lens = _random_paged(g, 3, 32, 4, 128, 16, lens, "bf16", "e4m3")
    q = (q.float() * 3.0e5).bfloat16()
    q[1, 5] = q[1, 5] * 1.0e-6  # one group's head tiny, another's huge
    q[2, 8:16] = 0.0  # a whole group of zeros
    ks, vs, scale = 1.0e-6, 0.013, 1.0 / math.sqrt(128)
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), oracle.E4M3, tables, lens, scale,
                               k_scale=ks, v_scale=vs)
    for path in (2, 3):
        pkv.set_kernel_path(path)
        got = _run_decode(pkv, q, kc, vc, tables, lens, scale, -1, ks, vs)
        assert_attention_close(got, want, TOL["e4m3"])


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_decode_tensor_core_e4m3_peaked_softmax(kernel_path, act):
    """Scores spread over tens of units: the weights span many orders of
    magnitude, and the small ones must still count (P's low E4M3 part)."""
    pkv = kernel_path
    g = _gen(92)
    lens = [33, 511, 1024, 1700]
    q, kc, vc, tables, lens = _random_paged(g, 4, 32, 4, 128, 32, lens, act, "e4m3")
    ks, vs, scale = 0.1, 0.013, 1.0 / math.sqrt(128)  # scores with a standard deviation near 10
    want = oracle.paged_decode(bits(q), ACT_CODE[DT[act]], bits(kc), bits(vc), oracle.E4M3, tables, lens, scale,
                               k_scale=ks, v_scale=vs)
    for path in (2, 3):
        pkv.set_kernel_path(path)
        got = _run_decode(pkv, q, kc, vc, tables, lens, scale, -1, ks, vs)
        assert_attention_close(got, want, TOL["e4m3"])


@pytest.mark.parametrize("path", [1, 3])
def test_decode_split_k_merge_many_rows(kernel_path, path):
    """4096 (sequence, query head) rows, so the merge takes one warp per row;
    1, 16, 17, 32, 33 and 35 partitions cover its 16-wide batch, the tail
    after it and the fallback beyond 32 (partitions of 64 tokens)."""
    pkv = kernel_path
    g = _gen(93)
    B, Hq, Hkv, bs = 64, 64, 8, 16
    lens = torch.randint(1, 2241, (B,), generator=g).numpy()
    lens[:8] = [1, 64, 1024, 1025, 2048, 2049, 2240, 63]
    q, kc, vc, tables, lens = _random_paged(g, B, Hq, Hkv, 128, bs, lens, "bf16", "bf16")
    scale = 1.0 / math.sqrt(128)
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), oracle.BF16, tables, lens, scale)
    pkv.set_kernel_path(path)
    got = _run_decode(pkv, q, kc, vc, tables, lens, scale, 64)
    assert_attention_close(got, want, TOL["bf16"])


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("path", [1, 2, 3])
def test_decode_ignores_unwritten_slots(kernel_path, path, D):
    """NaN in the never-written slots of each sequence's last block does not reach the output."""
    pkv = kernel_path
    g = _gen(77 + D)
    lens = [5, 37, 130, 300]
    q, kc, vc, tables, lens = _random_paged(g, 4, 16, 4, D, 16, lens, "bf16", "bf16")
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), oracle.BF16, tables, lens, 0.09)
    for b, L in enumerate(lens):
        last = int(tables[b, (L - 1) // 16])
        kc[last, :, L % 16 or 16:] = float("nan")
        vc[last, :, L % 16 or 16:] = float("nan")
    pkv.set_kernel_path(path)
    got = _run_decode(pkv, q, kc, vc, tables, lens, 0.09, -1)
    assert_attention_close(got, want, TOL["bf16"])


@pytest.mark.parametrize("path", [1, 2, 3])
def test_decode_e4m3_ignores_unwritten_slots(kernel_path, path):
    """NaN codes in the never-written slots of an E4M3 cache's last blocks do not reach the output."""
    pkv = kernel_path
    g = _gen(78)
    lens = [5, 37, 130, 300]
    q, kc, vc, tables, lens = _random_paged(g, 4, 32, 4, 128, 16, lens, "bf16", "e4m3")
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), oracle.E4M3, tables, lens, 0.09,
                               k_scale=0.02, v_scale=0.01)
    for b, L in enumerate(lens):
        last = int(tables[b, (L - 1) // 16])
        kc[last, :, L % 16 or 16:] = 0x7F  # E4M3 NaN
        vc[last, :, L % 16 or 16:] = 0xFF
    pkv.set_kernel_path(path)
    got = _run_decode(pkv, q, kc, vc, tables, lens, 0.09, -1, 0.02, 0.01)
    assert_attention_close(got, want, TOL["e4m3"])


def test_tensor_path_refuses_unsupported_shapes(kernel_path):
    pkv = kernel_path
    g = _gen(4)
    q, kc, vc, tables, lens = _random_paged(g, 2, 8, 8, 128, 16, [20, 40], "bf16", "bf16")  # group 1
    pkv.set_kernel_path(pkv.PATH_TENSOR)
    with pytest.raises(pkv.PagedKVError):
        _run_decode(pkv, q, kc, vc, tables, lens, 0.1, -1)
    # head_dim 64: an odd number of kv heads has no pairs; an E4M3 cache is not served
    q, kc, vc, tables, lens = _random_paged(g, 2, 12, 3, 64, 16, [20, 40], "bf16", "bf16")
    with pytest.raises(pkv.PagedKVError):
        _run_decode(pkv, q, kc, vc, tables, lens, 0.1, -1)
    q, kc, vc, tables, lens = _random_paged(g, 2, 16, 4, 64, 16, [20, 40], "bf16", "e4m3")
    with pytest.raises(pkv.PagedKVError):
        _run_decode(pkv, q, kc, vc, tables, lens, 0.1, -1, 0.02, 0.02)
    with pytest.raises(ValueError):
        pkv.set_kernel_path(9)


def test_bounded_wait_reports_timeout_and_context_survives(kernel_path):
    """A wait on a barrier nothing arrives at gives up after its limit and sets
    the timeout bit; the context stays usable for the next decode."""
    pkv = kernel_path
    pkv.device_error(reset=True)
    pkv.selftest_wait_timeout(2000)  # 2 ms instead of the kernels' 2 s
    assert pkv.device_error(reset=True) == pkv.DEV_WAIT_TIMEOUT
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, 4, 64, generator=g).half().cuda()
    kc = torch.randn(4, 4, 16, 64, generator=g).half().cuda()
    vc = torch.randn(4, 4, 16, 64, generator=g).half().cuda()
    tables = torch.tensor([[0, 1], [3, 2]], dtype=torch.int32).cuda()
    lens = torch.tensor([20, 32], dtype=torch.int32).cuda()
    out = pkv.paged_attention_decode(q, kc, vc, tables, lens, 0.125)
    torch.cuda.synchronize()
    assert pkv.device_error(reset=True) == 0
    want = oracle.paged_decode(bits(q.cpu()), oracle.F16, bits(kc.cpu()), bits(vc.cpu()), oracle.F16,
                               tables.cpu().numpy(), lens.cpu().numpy(), 0.125)
    assert np.abs(out.float().cpu().numpy() - want).max() <= TOL["f16"]


@pytest.mark.parametrize("path", [1, 3])
def test_output_to_pinned_host_memory(kernel_path, path):
    """out in pinned host memory: the kernels (partition, tensor-core and merge)
    store the result over the host link; it equals the device-memory output."""
    pkv = kernel_path
    pkv.set_kernel_path(path)
    g = torch.Generator().manual_seed(17 + path)
    B, Hq, Hkv, D, bs = 5, 32, 4, 128, 16
    lens = torch.tensor([1, 100, 700, 1500, 2000], dtype=torch.int32)
    maxb = -(-int(lens.max()) // bs)
    NB = B * maxb
    tables = torch.randperm(NB, generator=g)[: B * maxb].reshape(B, maxb).to(torch.int32)
    q = torch.randn(B, Hq, D, generator=g).bfloat16().cuda()
    kc = torch.randn(NB, Hkv, bs, D, generator=g).bfloat16().cuda()
    vc = torch.randn(NB, Hkv, bs, D, generator=g).bfloat16().cuda()
    t_d, l_d = tables.cuda(), lens.cuda()
    want = pkv.paged_attention_decode(q, kc, vc, t_d, l_d, 0.088, partition_size=512)
    host = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16).pin_memory()
    got = pkv.paged_attention_decode(q, kc, vc, t_d, l_d, 0.088, out=host, partition_size=512)
    torch.cuda.synchronize()
    assert got is host and torch.equal(host, want.cpu())


@pytest.mark.parametrize("fused", [False, True])
def test_decode_plan_matches_the_calls(kernel_path, fused):
    """DecodePlan.run() gives the same bits as the one-shot call, and sees new
    contents of its fixed tensors between runs."""
    pkv = kernel_path
    g = _gen(94)
    lens = [40, 300, 1025, 7]
    q, kc, vc, tables, lens = _random_paged(g, 4, 32, 4, 128, 16, lens, "bf16", "bf16")
    q, kc, vc = q.cuda(), kc.cuda(), vc.cuda()
    tab, ln = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    kw = {}
    if fused:
        kw = dict(k_new=torch.randn(4, 4, 128, generator=g).bfloat16().cuda(),
                  v_new=torch.randn(4, 4, 128, generator=g).bfloat16().cuda(),
                  slot_mapping=torch.tensor([int(tables[b, (L - 1) // 16]) * 16 + (L - 1) % 16
                                             for b, L in enumerate(lens)], dtype=torch.int64).cuda())
    out = torch.empty_like(q)
    pkv.set_kernel_path(pkv.PATH_AUTO)
    plan = pkv.DecodePlan(q, kc, vc, tab, ln, 0.088, out=out, **kw)
    for step in range(2):
        if step == 1:
            q.copy_(torch.randn(q.shape, generator=g).bfloat16())  # new queries in the same storage
        kc2, vc2 = kc.clone(), vc.clone()
        got = plan.run().clone()
        if fused:
            want = pkv.paged_attention_decode_append(q, kw["k_new"], kw["v_new"], kw["slot_mapping"], kc2, vc2, tab,
                                                     ln, 0.088)
        else:
            want = pkv.paged_attention_decode(q, kc2, vc2, tab, ln, 0.088)
        torch.cuda.synchronize()
        assert torch.equal(got, want)


@pytest.mark.parametrize("cache", ["bf16", "e4m3"])
def test_decode_tensor_core_many_rows(kernel_path, cache):
    """720 sequences: the per-row tables leave room for only two 32 KB stages
    (16-bit cache, more than 292 rows) or four 16 KB stages (E4M3, more than
    698 rows) at two CTAs per SM, so the smaller rings run."""
    pkv = kernel_path
    g = _gen(95)
    B = 720
    lens = torch.randint(1, 201, (B,), generator=g).numpy()
    q, kc, vc, tables, lens = _random_paged(g, B, 32, 4, 128, 16, lens, "bf16", cache)
    scale = 1.0 / math.sqrt(128)
    ks, vs = (0.021, 0.013) if cache == "e4m3" else (None, None)
    code = oracle.E4M3 if cache == "e4m3" else oracle.BF16
    want = oracle.paged_decode(bits(q), oracle.BF16, bits(kc), bits(vc), code, tables, lens, scale,
                               **({"k_scale": ks, "v_scale": vs} if ks else {}))
    pkv.set_kernel_path(pkv.PATH_TENSOR_2CTA)
    got = _run_decode(pkv, q, kc, vc, tables, lens, scale, 128, ks, vs)
    assert_attention_close(got, want, TOL[cache])


def test_decode_tensor_core_more_than_one_launch_of_rows(kernel_path):
    """More sequences than one tensor-core launch serves (2048 table rows):
    the library runs consecutive chunks of sequences, each its own persistent
    launch, then one merge.  2500 sequences with the new token fused in, a
    few long enough to split into several partitions, every output against
    the oracle and every appended row bit for bit."""
    pkv = kernel_path
    g = _gen(2500)
    B, Hq, Hkv, D, bs = 2500, 32, 8, 128, 16
    lens = torch.randint(1, 96, (B,), generator=g).numpy()
    lens[[0, 1047, 2047, 2048, 2499]] = [1500, 700, 513, 1100, 2000]  # split-K rows on both sides of the cut
    q, kc, vc, tables, lens = _random_paged(g, B, Hq, Hkv, D, bs, lens, "bf16", "bf16")
    k_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    slots = np.array([oracle.slot_of(tables[b], int(lens[b]) - 1, bs) for b in range(B)], np.int64)
    rk, rv = bits(kc).copy(), bits(vc).copy()
    oracle.append(bits(k_new), bits(v_new), oracle.BF16, slots, rk, rv, oracle.BF16)
    scale = 1.0 / math.sqrt(D)
    want = oracle.paged_decode(bits(q), oracle.BF16, rk, rv, oracle.BF16, tables, lens, scale)
    dk, dv = kc.cuda(), vc.cuda()
    assert pkv.resolve_partition_size(B, Hq, Hkv, D, tables.shape[1], bs, -1) == 512  # the tensor-core choice
    got = pkv.paged_attention_decode_append(q.cuda(), k_new.cuda(), v_new.cuda(), torch.from_numpy(slots).cuda(),
                                            dk, dv, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                                            scale)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dk), rk) and np.array_equal(bits(dv), rv)
    assert_attention_close(got, want, TOL["bf16"])
    # per-(sequence, kv head) tables: 300 x 8 = 2400 rows, also more than one launch
    Bs = 300
    sel = np.repeat(tables[:Bs, None, :], Hkv, axis=1).copy()
    slen = np.repeat(lens[:Bs, None], Hkv, axis=1).astype(np.int32)
    out = pkv.paged_attention_decode_sparse(q[:Bs].contiguous().cuda(), dk, dv, torch.from_numpy(sel).cuda(),
                                            torch.from_numpy(slen).cuda(), scale)
    torch.cuda.synchronize()
    want_s = oracle.sparse_decode(bits(q[:Bs]), oracle.BF16, rk, rv, oracle.BF16, sel, slen, scale)
    assert_attention_close(out, want_s, TOL["bf16"])
