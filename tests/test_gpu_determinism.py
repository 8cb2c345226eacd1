"""Run-to-run determinism: the same step on the same inputs gives the same bits.

Every kernel of the step reduces in a fixed order (no floating-point atomics
on results): the indexer scan, the Top-K selection, the block pool, the
compression GEMM's split-K sum, the packing and the attention (including the
cluster merge of decode).  Two runs of a layer group must agree bit for bit in
indices, counts, pools, outputs, lse and the bytes the step packs.
"""
import pytest
import torch

from compressed_sparse_attention_05_gb300 import abi, build, harness
from csa2_inputs import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()


def _decode():
    return WL.decode_128k(B=4, L=4 * 30000 + 1)


def _decode_fp8kv():
    wl = WL.decode_fp8kv_128k(B=4, L=4 * 30000 + 1)
    return wl


def _prefill():
    return WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)


def _hierarchical():
    return WL.hierarchical_1m(B=2, L=4 * 40000 + 2)


def _snapshot(g):
    out = []
    for t in [*g.idx, *g.cnt, g.pool, g.pool_cnt, g.kv_codes, g.kv_scales, g.idx_k]:
        out.append(t.clone())
    for t in [*g.O, *g.lse]:
        out.append(t.view(torch.int32).clone())   # bits, NaN-safe
    return out


@pytest.mark.parametrize("make", [_decode, _decode_fp8kv, _prefill, _hierarchical],
                         ids=["decode", "decode_fp8kv", "prefill", "hierarchical"])
def test_step_bits_repeat(make):
    wl = make()
    g = harness.LayerGroup(wl)
    g.step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    first = _snapshot(g)
    for t in [*g.O, *g.lse]:
        t.fill_(float("nan"))
    for t in [*g.idx, *g.cnt, g.pool, g.pool_cnt]:
        t.fill_(-7)
    g.step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    second = _snapshot(g)
    for i, (a, b) in enumerate(zip(first, second)):
        assert torch.equal(a, b), f"tensor {i} differs between two runs of the same step"
