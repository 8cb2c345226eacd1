"""csa2_index_topk_noalloc against csa2_index_topk.

The no-allocation variant serves callers that cannot allocate device memory
(for example while a CUDA graph is being captured, or on a serving thread that
must never wait on the allocator): its scratch is a fixed array inside the
library instead of a caller workspace.  It must give exactly the indices,
counts and pools of the workspace entry point (same kernels, same inputs:
index work is compared bit for bit), call after call, since every call
reuses the same array.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
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


def _outputs(wl, with_pool):
    dev = "cuda"
    rows = (wl.B, wl.Tq)
    idx = torch.full((*rows, wl.K), -7, dtype=torch.int32, device=dev)
    cnt = torch.full(rows, -7, dtype=torch.int32, device=dev)
    pool = torch.full((*rows, wl.pool_blocks), -7, dtype=torch.int32, device=dev) if with_pool else None
    pcnt = torch.full(rows, -7, dtype=torch.int32, device=dev) if with_pool else None
    return idx, cnt, pool, pcnt


def _same(a, b):
    return all((x is None and y is None) or torch.equal(x, y) for x, y in zip(a, b))


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    wl = WL.hierarchical_1m(B=3, L=4 * 20000 + 2)       # Full layer with the 2,048-block pool
    g = harness.LayerGroup(wl)
    dims, cache = g.dims(), g.cache()
    need = abi.csa2_index_topk_workspace_size(dims, g.max_entries)
    assert 0 < need <= abi.csa2_index_topk_noalloc_capacity()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    # Full mode with pool, through the caller-workspace entry point
    ref = _outputs(wl, True)
    abi.csa2_index_topk(dims, cache, g.idx_q[0], g.idx_w[0], g.q_pos, ref[0], ref[1], g.max_entries, ws,
                        out_pool=ref[2], out_pool_cnt=ref[3])
    # Reindex mode over that pool
    ref_x = _outputs(wl, False)
    abi.csa2_index_topk(dims, cache, g.idx_q[1], g.idx_w[1], g.q_pos, ref_x[0], ref_x[1], g.max_entries, ws,
                        pool=ref[2], pool_cnt=ref[3])
    torch.cuda.synchronize()
    assert int(ref[1].min()) == wl.K and int(ref[3].min()) == wl.pool_blocks

    for _ in range(2):   # two calls in a row reuse the same fixed scratch
        got = _outputs(wl, True)
        abi.csa2_index_topk_noalloc(dims, cache, g.idx_q[0], g.idx_w[0], g.q_pos, got[0], got[1], g.max_entries,
                                    out_pool=got[2], out_pool_cnt=got[3])
        got_x = _outputs(wl, False)
        abi.csa2_index_topk_noalloc(dims, cache, g.idx_q[1], g.idx_w[1], g.q_pos, got_x[0], got_x[1],
                                    g.max_entries, pool=got[2], pool_cnt=got[3])
        torch.cuda.synchronize()
        assert _same(got, ref)
        assert _same(got_x, ref_x)
    assert abi.csa2_get_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    wl = WL.decode_128k(B=64, L=1048576)
    dims = abi.Dims(B=wl.B, Tq=1, d=512, r=64, Hq=64, Hi=8, Di=128, idx_dtype=abi.CSA2_BF16, K=512, W=128,
                    max_pages=4096, n_pool_blocks=2048, pool_block=8, swa_cap=128)
    assert abi.csa2_index_topk_workspace_size(dims, 262144) > abi.csa2_index_topk_noalloc_capacity()
    fake = 1 << 20
    cache = abi.Cache(kv_codes=fake, kv_scales=fake, idx_k=fake, page_table=fake, n_entries=fake, n_pages=1)
    rc = abi.lib().csa2_index_topk_noalloc(abi.C.byref(dims), abi.C.byref(cache), fake, fake, fake, None, None,
                                           fake, fake, None, None, 262144, None)
    assert rc == 4
    assert "8 MiB" in abi.lib().csa2_last_error().decode()
