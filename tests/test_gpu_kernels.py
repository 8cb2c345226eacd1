"""Bit-exact parity of the packing, Top-K and pooling kernels with the oracle,
on given fp32 arrays (tiles, ragged tails, ties, zero groups, saturation)."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_05_gb300 import abi, build
from oracle import formats as F
from oracle import indexer as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()
    yield
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0


def _mx_rows():
    g = torch.Generator().manual_seed(11)
    rows = [torch.randn(3000, 512, generator=g) * torch.tensor([1e-4, 1e-2, 1, 7, 300, 1e5]).repeat(500)[:, None]]
    # tie values: with amax = 6 the scale is exactly 1, so x / s is the value itself
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 3.0, 5.5, 0.0])
    t = torch.zeros(64, 512)
    for i in range(64):
        pick = torch.randint(0, len(mids), (15,), generator=g)
        grp = torch.cat([torch.tensor([6.0]), mids[pick] * (1 - 2 * (i % 2))])
        t[i] = grp.repeat(32)
    rows.append(t)
    z = torch.zeros(8, 512)
    z[1, 3] = -1e-30
    z[2, :16] = -0.0
    z[3] = 1e38
    rows.append(z)
    return torch.cat(rows).float().contiguous()


def test_pack_mxfp4_bit_exact():
    x = _mx_rows()
    codes = torch.empty(x.shape[0], 256, dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.shape[0], 32, dtype=torch.uint8, device="cuda")
    abi.csa2_pack_mxfp4_f32(x.cuda(), codes, scales)
    rc, rs = F.mxfp4_pack(x.numpy())
    gs, gc = scales.cpu().numpy(), codes.cpu().numpy()
    assert np.array_equal(gs, rs)
    bad = np.argwhere(gc != rc)
    if len(bad):
        r, byte = bad[0]
        grp = byte // 8
        xs = x[r, grp * 16:(grp + 1) * 16].numpy()
        raise AssertionError(f"{len(bad)} code bytes differ; first at row {r} byte {byte}: gpu {gc[r, byte]:#04x} "
                             f"oracle {rc[r, byte]:#04x}; scale {rs[r, grp]:#04x}; group {xs.tolist()}")


def test_pack_mxfp4_d64_and_ragged_rows():
    g = torch.Generator().manual_seed(12)
    x = (torch.randn(777, 64, generator=g) * 3).contiguous()
    codes = torch.empty(777, 32, dtype=torch.uint8, device="cuda")
    scales = torch.empty(777, 4, dtype=torch.uint8, device="cuda")
    abi.csa2_pack_mxfp4_f32(x.cuda(), codes, scales)
    rc, rs = F.mxfp4_pack(x.numpy())
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)


def test_unpack_mxfp4_exact():
    g = torch.Generator().manual_seed(13)
    codes = torch.randint(0, 256, (300, 256), generator=g, dtype=torch.uint8)
    scales = torch.randint(0, 127, (300, 32), generator=g, dtype=torch.uint8)   # finite E4M3 codes
    out = torch.empty(300, 512, dtype=torch.bfloat16, device="cuda")
    abi.csa2_unpack_mxfp4_bf16(codes.cuda(), scales.cuda(), out)
    ref = F.mxfp4_unpack(codes.numpy(), scales.numpy())
    assert np.array_equal(out.float().cpu().double().numpy(), ref)


def test_pack_fp8_bit_exact():
    g = torch.Generator().manual_seed(14)
    x = torch.randn(2000, 512, generator=g) * torch.tensor([1e-3, 1, 50, 1e4]).repeat(500)[:, None]
    t = torch.zeros(40, 512)
    fin = [c for c in range(1, 126)]
    for i in range(40):   # amax 448 -> scale 1: x / s hits E4M3 midpoints exactly
        a = torch.tensor([F.E4M3_TABLE[c] for c in fin])
        b = torch.tensor([F.E4M3_TABLE[c + 1] for c in fin])
        mid = ((a + b) / 2)[torch.randint(0, len(fin), (511,), generator=g)]
        t[i] = torch.cat([torch.tensor([448.0]), mid * (1 - 2 * (i % 2))])
    x = torch.cat([x, t, torch.zeros(3, 512)]).float().contiguous()
    codes = torch.empty(x.shape[0], 512, dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.shape[0], dtype=torch.float32, device="cuda")
    abi.csa2_pack_swa_fp8(x.cuda(), codes, scales)
    rc, rs = F.fp8_pack(x.numpy())
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), rc)


def _score_rows():
    g = torch.Generator().manual_seed(15)
    rows, n_valid = [], []
    stride = 40000
    # "const" and "narrow" put more than 4,096 entries in the threshold bin of the
    # 11-bit key histogram, which takes the whole-row radix path
    for n, kind in [(40000, "normal"), (33333, "ties"), (5000, "ties2"), (512, "normal"), (300, "normal"),
                    (0, "normal"), (1, "normal"), (513, "zeros"), (20000, "neg"), (16385, "ties"),
                    (40000, "const"), (30000, "narrow"), (32768, "tiesK"), (32768, "tiesK2")]:
        if kind == "normal":
            r = torch.randn(stride, generator=g)
        elif kind == "ties":
            r = torch.randint(-20, 20, (stride,), generator=g).float() * 0.5
        elif kind == "ties2":
            r = torch.randint(0, 3, (stride,), generator=g).float()
        elif kind == "zeros":
            r = torch.zeros(stride)
            r[torch.randperm(stride, generator=g)[:200]] = -0.0
            r[5] = 1.0
        elif kind == "const":
            r = torch.full((stride,), 2.5)
        elif kind == "narrow":
            r = 1.0 + torch.rand(stride, generator=g) * 0.2
        elif kind.startswith("tiesK"):
            # 300 copies of the 401st (1,901st) largest value spread over the row: the
            # Top-512 (Top-2048) takes some of the ties, by lower index
            r = torch.randn(stride, generator=g)
            v = torch.sort(r[:n], descending=True).values[400 if kind == "tiesK" else 1900]
            below = torch.nonzero(r[:n] < v).flatten()
            r[below[torch.randperm(len(below), generator=g)[:300]]] = v
        else:
            r = -torch.rand(stride, generator=g) * 1e-30 - 1e-38
        r[n:] = float("nan")   # never read: beyond the valid count
        rows.append(r)
        n_valid.append(n)
    return torch.stack(rows).contiguous(), torch.tensor(n_valid, dtype=torch.int32)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("k", [512, 16, 2048, 1])
def test_topk_bit_exact(k, split):
    s, nv = _score_rows()
    rows = s.shape[0]
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    ws = None
    if split:   # many CTAs per row
        ws = torch.empty(abi.csa2_topk_workspace_size(rows, s.shape[1], k), dtype=torch.uint8, device="cuda")
    abi.csa2_topk_f32(s.cuda(), nv.cuda(), k, idx, cnt, ws=ws)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(rows):
        ref = I.topk(s[r, :nv[r]].numpy(), k)
        assert cnt[r] == len(ref), r
        assert np.array_equal(idx[r, :cnt[r]], ref), r
        assert np.all(idx[r, cnt[r]:] == -1)


@pytest.mark.parametrize("k", [512, 16])
def test_topk_bit_exact_unaligned_rows(k):
    """Rows that do not start on a 16-byte boundary (odd stride) take the
    scalar-load pass; same selection rule."""
    s, nv = _score_rows()
    s = torch.nn.functional.pad(s, (0, 1), value=float("nan")).contiguous()   # stride 40,001
    rows = s.shape[0]
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    abi.csa2_topk_f32(s.cuda(), nv.cuda(), k, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(rows):
        ref = I.topk(s[r, :nv[r]].numpy(), k)
        assert cnt[r] == len(ref), r
        assert np.array_equal(idx[r, :cnt[r]], ref), r
        assert np.all(idx[r, cnt[r]:] == -1)


@pytest.mark.parametrize("stride", [32768, 20001])
@pytest.mark.parametrize("k", [512, 2048])
def test_topk_bit_exact_rows_in_registers(stride, k):
    """Few rows of at most 32,768 entries: one 1024-thread CTA per row holds
    the row in registers (histogram built from them, one read)."""
    s, nv = _score_rows()
    s = s[:, :stride].contiguous() if stride <= s.shape[1] else s
    nv = torch.clamp(nv, max=stride)
    rows = s.shape[0]
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    abi.csa2_topk_f32(s.cuda(), nv.cuda(), k, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(rows):
        ref = I.topk(s[r, :nv[r]].numpy(), k)
        assert cnt[r] == len(ref), r
        assert np.array_equal(idx[r, :cnt[r]], ref), r
        assert np.all(idx[r, cnt[r]:] == -1)


@pytest.mark.parametrize("stride", [20000, 20001, 32768])
@pytest.mark.parametrize("k", [512, 2048])
def test_topk_bit_exact_with_histogram(stride, k):
    """Row histograms given (the workspace path builds them first): rows of
    8,193..32,768 entries are spread over a cluster of CTAs per row for K = 512
    and taken by one CTA per row for K = 2,048."""
    s, nv = _score_rows()
    s = s[:, :stride].contiguous() if stride <= s.shape[1] else torch.nn.functional.pad(
        s, (0, stride - s.shape[1]), value=float("nan")).contiguous()
    nv = torch.clamp(nv, max=stride)
    rows = s.shape[0]
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(abi.csa2_topk_workspace_size(rows, stride, k), dtype=torch.uint8, device="cuda")
    abi.csa2_topk_f32(s.cuda(), nv.cuda(), k, idx, cnt, ws=ws)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(rows):
        ref = I.topk(s[r, :nv[r]].numpy(), k)
        assert cnt[r] == len(ref), r
        assert np.array_equal(idx[r, :cnt[r]], ref), r
        assert np.all(idx[r, cnt[r]:] == -1)


def _many_short_rows(stride):
    """320 rows (more than twice the SM count) of at most 32,768 entries: the
    many-short-rows path (sampled lower bound, candidates only; the whole-row
    radix fallback for rows of equal or crowded scores), vectorised when rows
    are 16-byte aligned (strides 16,384, 4,000 and 32,768)."""
    g = torch.Generator().manual_seed(16)
    kinds = ["normal", "ties", "ties2", "zeros", "neg", "const", "narrow", "normal"]
    rows, n_valid = [], []
    for r in range(320):
        kind = kinds[r % len(kinds)]
        n = [stride, stride - 3, 513, 512, 300, 0, 1, 4097, stride // 2 + 1][r % 9]
        if kind == "normal":
            x = torch.randn(stride, generator=g)
        elif kind == "ties":
            x = torch.randint(-20, 20, (stride,), generator=g).float() * 0.5
        elif kind == "ties2":
            x = torch.randint(0, 3, (stride,), generator=g).float()
        elif kind == "zeros":
            x = torch.zeros(stride)
            x[torch.randperm(stride, generator=g)[:200]] = -0.0
            x[5] = 1.0
        elif kind == "const":
            x = torch.full((stride,), 2.5)
        elif kind == "narrow":
            x = 1.0 + torch.rand(stride, generator=g) * 0.2
        else:
            x = -torch.rand(stride, generator=g) * 1e-30 - 1e-38
        x[n:] = float("nan")   # never read: beyond the valid count
        rows.append(x)
        n_valid.append(n)
    return torch.stack(rows).contiguous(), torch.tensor(n_valid, dtype=torch.int32)


@pytest.mark.parametrize("stride", [16384, 4000, 12001, 32768])
@pytest.mark.parametrize("k", [512, 7])
def test_topk_bit_exact_many_short_rows(stride, k):
    s, nv = _many_short_rows(stride)
    rows = s.shape[0]
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    abi.csa2_topk_f32(s.cuda(), nv.cuda(), k, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(rows):
        ref = I.topk(s[r, :nv[r]].numpy(), k)
        assert cnt[r] == len(ref), r
        assert np.array_equal(idx[r, :cnt[r]], ref), r
        assert np.all(idx[r, cnt[r]:] == -1)


def test_block_pool_bit_exact():
    s, nv = _score_rows()
    rows = s.shape[0]
    nb = 2048
    pool = torch.full((rows, nb), -5, dtype=torch.int32, device="cuda")
    pcnt = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    bm = torch.full((rows, (s.shape[1] + 7) // 8), float("nan"), device="cuda")
    abi.csa2_block_pool_f32(s.cuda(), nv.cuda(), 8, nb, pool, pcnt, bm)
    pool, pcnt, bm = pool.cpu().numpy(), pcnt.cpu().numpy(), bm.cpu().numpy()
    for r in range(rows):
        n = int(nv[r])
        ref_bm = I.block_scores(s[r, :n].numpy(), 8)
        assert np.array_equal(bm[r, :len(ref_bm)].astype(np.float64), ref_bm), r
        ref = I.block_pool(s[r, :n].numpy(), nb, 8)
        assert pcnt[r] == len(ref) and np.array_equal(pool[r, :pcnt[r]], ref), r
        assert np.all(pool[r, pcnt[r]:] == -1)


def test_status_word_clean():
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
