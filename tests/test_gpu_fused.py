"""Fused append + decode: one launch gives the same cache bytes and the same
output bits as paged_kv_append followed by paged_attention_decode, and matches
the float64 oracle."""
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


CASES = [
    # act, cache, Hq, Hkv, D, bs, partition
    ("bf16", "bf16", 8, 8, 128, 16, -1),
    ("bf16", "bf16", 8, 8, 128, 16, 64),
    ("f16", "f16", 8, 8, 64, 32, 64),
    ("bf16", "e4m3", 4, 4, 128, 16, 128),
    ("bf16", "bf16", 32, 4, 128, 16, -1),   # tensor-core path
    ("f16", "f16", 32, 4, 128, 32, 128),    # tensor-core path
    ("bf16", "bf16", 16, 8, 128, 16, 64),   # group 2: CUDA-core path
    ("bf16", "e4m3", 32, 4, 128, 16, -1),   # tensor-core path, E4M3 cache
    ("f16", "e4m3", 32, 4, 128, 32, 128),   # tensor-core path, E4M3 cache
    ("bf16", "bf16", 32, 4, 64, 16, -1),    # tensor-core path, head_dim 64 (two kv heads per item)
    ("f16", "f16", 16, 2, 64, 32, 128),     # tensor-core path, head_dim 64, one pair
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_fused_equals_append_then_decode(pkv, case):
    act, cache, Hq, Hkv, D, bs, part = case
    g = torch.Generator().manual_seed(zlib.crc32(repr(case).encode()))
    ctx = [0, 15, 16, 63, 64, 127, 300, 1023, 2000]  # tokens already in the cache
    B = len(ctx)
    NB = sum(-(-(c + 1) // bs) for c in ctx) + 4
    fl = torch.randperm(NB, generator=g).numpy().astype(np.int32)
    ref = RefBlockManager(NB, bs, free_list=fl)
    for i, c in enumerate(ctx):
        ref.add_sequence(i, c)
    slots = np.array([ref.append_slot(i)[0] for i in range(B)], np.int64)
    slots[1] = -1  # sequence 1 has no new token this step
    lens = np.array([c + 1 for c in ctx], np.int32)
    lens[1] = ctx[1]
    maxb = max(len(t) for t in ref.tables.values())
    tables = np.zeros((B, maxb), np.int32)
    for i in range(B):
        tables[i, : len(ref.tables[i])] = ref.tables[i]
    q = torch.randn(B, Hq, D, generator=g).to(DT[act])
    k_new = torch.randn(B, Hkv, D, generator=g).to(DT[act])
    v_new = torch.randn(B, Hkv, D, generator=g).to(DT[act])
    if cache == "e4m3":
        kc = torch.randint(0, 256, (NB, Hkv, bs, D), dtype=torch.uint8, generator=g)
        kc[(kc & 0x7F) == 0x7F] = 0x30
        vc = kc.flip(0).contiguous()
        ks, vs = torch.tensor([0.021]), torch.tensor([0.013])
    else:
        kc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
        vc = torch.randn(NB, Hkv, bs, D, generator=g).to(DT[act])
        ks = vs = None
    dev = torch.device("cuda")
    cu = lambda t: None if t is None else t.to(dev)
    t_d, l_d, s_d = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev), torch.from_numpy(slots).to(dev)
    # separate launches
    ka, va = kc.to(dev), vc.to(dev)
    pkv.paged_kv_append(cu(k_new), cu(v_new), s_d, ka, va, cu(ks), cu(vs))
    out_a = pkv.paged_attention_decode(cu(q), ka, va, t_d, l_d, 0.1, k_scale=cu(ks), v_scale=cu(vs),
                                       partition_size=part)
    # fused
    kb, vb = kc.to(dev), vc.to(dev)
    out_b = pkv.paged_attention_decode_append(cu(q), cu(k_new), cu(v_new), s_d, kb, vb, t_d, l_d, 0.1,
                                              k_scale=cu(ks), v_scale=cu(vs), partition_size=part)
    torch.cuda.synchronize()
    assert torch.equal(ka, kb) and torch.equal(va, vb), "fused append wrote different cache bytes"
    assert torch.equal(out_a, out_b), "fused output differs from append + decode"
    code = oracle.E4M3 if cache == "e4m3" else ACT_CODE[DT[act]]
    want = oracle.paged_decode(bits(q), ACT_CODE[DT[act]], bits(kb), bits(vb), code, tables, lens, 0.1,
                               k_scale=float(ks) if ks is not None else 1.0,
                               v_scale=float(vs) if vs is not None else 1.0)
    assert_attention_close(out_b, want, TOL["e4m3" if cache == "e4m3" else act])
