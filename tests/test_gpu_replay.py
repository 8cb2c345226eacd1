"""SWA Bounded Replay ("DeepSeek-V4.1 架构解析" §03): window rows rebuilt from the
replayed tokens' hidden states by csa2_swa_replay, against the oracle's rows.

The codes are decided from the GEMM's fp32 sums and an fp32 RMSNorm, the
oracle's from float64: they agree except where the oracle's value lies within
the propagated error bound of an E4M3 rounding boundary, and such a flip moves
the code by one step (parity.check_fp8_after_gemm)."""
import numpy as np
import pytest
import torch

import parity
from compressed_sparse_attention_05_gb300 import abi, build
from oracle import replay as R

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()


def _np(t):
    return t.detach().cpu().double().numpy()


def _dims(B, d, r, swa_cap):
    return abi.Dims(B=B, Tq=1, d=d, r=r, Hq=4, Hi=4, Di=32, idx_dtype=abi.CSA2_BF16, K=16, W=128, max_pages=1,
                    n_pool_blocks=0, pool_block=8, swa_cap=swa_cap)


def _check_rows(cg, sg, hidden, W, gamma, ref, r, eps=1e-6):
    """Rows [n, d] of the GPU window against the oracle's rows ``ref`` (window_rows output)."""
    tau_c = parity.gemm_error_bound(hidden, W)
    tau_x = parity.latent_error_bound(ref["c"], tau_c, gamma, eps, r, ref["x"])
    parity.check_fp8_after_gemm(cg, sg, ref["x"], tau_x)


def _run(hidden, W, gamma, tok0, win_pos0, cap, d, r, eps=1e-6, base=10000.0):
    dev = "cuda"
    B, n_tok, H = hidden.shape
    codes = torch.full((B, cap, d), 0xEE, dtype=torch.uint8, device=dev)
    scales = torch.full((B, cap), -1.0, device=dev)
    pos0 = torch.tensor(win_pos0, dtype=torch.int32, device=dev)
    win = abi.Window(codes=codes.data_ptr(), scales=scales.data_ptr(), pos0=pos0.data_ptr())
    ws = torch.empty(max(256, abi.csa2_swa_replay_workspace_size(B, n_tok, H, d)), dtype=torch.uint8, device=dev)
    tp = torch.tensor(tok0, dtype=torch.int32, device=dev)
    abi.csa2_swa_replay(hidden.to(dev), W.to(dev), gamma.to(dev), eps, base, tp, _dims(B, d, r, cap), win, ws)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), abi.csa2_get_status()


# (512, 64, 256, 130): two row tiles, the second ragged; (512, 64, 4096, 128): the
# pages' hidden width; (64, 16, 128, 37): the small latent (mma.sync GEMM)
@pytest.mark.parametrize("d,r,H,n_tok", [(512, 64, 256, 130), (512, 64, 4096, 128), (64, 16, 128, 37)])
def test_swa_replay_rows_match_oracle(d, r, H, n_tok):
    g = torch.Generator().manual_seed(31)
    B = 3
    hidden = torch.randn(B, n_tok, H, generator=g).to(torch.bfloat16)
    hidden[0, 5, 3] = 10.0
    W = (torch.randn(d, H, generator=g) * 0.02).to(torch.bfloat16)
    gamma = 1.0 + 0.05 * torch.randn(d, generator=g)
    tok0 = [4000, 7, 131000]
    off = [3, 0, 5]                                   # window rows before the replayed ones
    cap = n_tok + 8
    cg, sg, status = _run(hidden, W, gamma, tok0, [t - o for t, o in zip(tok0, off)], cap, d, r)
    assert status == 0
    for b in range(B):
        ref = R.window_rows(_np(hidden[b]), _np(W), _np(gamma), 1e-6, r, 10000.0, tok0[b])
        rows = slice(off[b], off[b] + n_tok)
        _check_rows(cg[b, rows], sg[b, rows], _np(hidden[b]), _np(W), _np(gamma), ref, r)
        # the rows around the replayed ones are not written
        assert np.all(cg[b, :off[b]] == 0xEE) and np.all(cg[b, off[b] + n_tok:] == 0xEE)
        assert np.all(sg[b, :off[b]] == -1.0) and np.all(sg[b, off[b] + n_tok:] == -1.0)


def test_swa_replay_rows_outside_the_window_are_skipped_and_flagged():
    # window rows 0..5 hold raw positions 102..107; tokens 100, 101 and 108, 109 fall outside
    g = torch.Generator().manual_seed(32)
    d, r, H, n_tok = 512, 64, 128, 10
    hidden = torch.randn(1, n_tok, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(d, H, generator=g) * 0.02).to(torch.bfloat16)
    gamma = torch.ones(d)
    cg, sg, status = _run(hidden, W, gamma, [100], [102], 6, d, r)
    assert status == abi.STATUS_BAD_COUNT
    ref = R.window_rows(_np(hidden[0]), _np(W), _np(gamma), 1e-6, r, 10000.0, 100)
    sub = {k: v[2:8] for k, v in ref.items()}
    _check_rows(cg[0], sg[0], _np(hidden[0])[2:8], _np(W), _np(gamma), sub, r)
