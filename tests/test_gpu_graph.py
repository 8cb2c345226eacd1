"""A layer step captured in a CUDA graph gives the same bits as direct launches.

csa2_layer launches its kernels with programmatic stream serialisation and
allocates nothing, so a serving loop can capture a step once and replay it.
The captured decode and prefill (with compression) steps must reproduce the
directly launched step's indices, counts, outputs and lse bit for bit.
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


def _prefill():
    return WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)


def _outputs(g):
    return [t.clone() for t in [*g.idx, *g.cnt]] + [t.view(torch.int32).clone() for t in [*g.O, *g.lse]]


@pytest.mark.parametrize("make", [_decode, _prefill], ids=["decode", "prefill"])
def test_captured_step_matches_direct(make):
    g = harness.LayerGroup(make())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.step(stream=s)          # warm-up: kernel attributes, tensor maps, symbol addresses
    torch.cuda.synchronize()
    direct = _outputs(g)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.step(stream=s)
    for t in [*g.O, *g.lse]:
        t.fill_(float("nan"))
    for t in [*g.idx, *g.cnt]:
        t.fill_(-7)
    graph.replay()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    for i, (a, b) in enumerate(zip(direct, _outputs(g))):
        assert torch.equal(a, b), f"tensor {i} differs between the captured and the direct step"
