"""Attention on bf16 operands outside fp16's range (reading R11 of include/csa2.h).

The kernels carry Q and the dequantised window rows in fp16 after a power of
two per head (Q) or per window row (scales outside [2^-8, 2^7]); every bf16
value keeps all its bits.  Checked against the float64 oracle on the same
operands, with Q heads reaching |x| ~ 4e5 (beyond fp16's 65504) and ~1e-6
(below its normal range), window rows whose largest value is ~3e5 or ~1e-6,
and tokens that attend to tiny window rows only.
"""
import math

import numpy as np
import pytest
import torch

import parity
from compressed_sparse_attention_05_gb300 import abi, build, harness
from csa2_inputs import workloads as WL
from oracle import attention as A
from oracle import formats as F
from oracle import layer as OL
from layer_check import Operands

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()


def _decode_small():
    wl = WL.decode_128k(B=3, L=4096)
    wl.t_first = [20001, 4098, 777]
    wl.name = "decode_small"
    return wl


def _tiny():
    return WL.tiny()


@pytest.mark.parametrize("make", [_decode_small, _tiny], ids=["d512", "d64"])
def test_attention_operands_beyond_fp16_range(make):
    wl = make()
    g = harness.LayerGroup(wl)
    g.step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    dev = g.Q[0].device
    B, Tq, Hq, d = wl.B, wl.Tq, wl.Hq, wl.d
    rows = [(b, i) for b in range(B) for i in ([0] if Tq == 1 else [0, 5, Tq - 1])]

    # Q: head 0 scaled to ~4e5, head 1 to ~1e-6, head 2 alternating 1e4 / 1e-4
    Q = g.Q[0].clone()
    Q[:, :, 0] = (Q[:, :, 0].float() * 1e5).to(torch.bfloat16)
    Q[:, :, 1] = (Q[:, :, 1].float() * 1e-6).to(torch.bfloat16)
    alt = torch.where(torch.arange(d, device=dev) % 2 == 0, 1e4, 1e-4)
    Q[:, :, 2] = (Q[:, :, 2].float() * alt).to(torch.bfloat16)

    # window rows: each sampled token's own row ~3e5, the row before it ~1e-6; the last
    # sampled token attends to its window rows only (no selected entries), all ~1e-6
    cnt = g.cnt[0].clone()
    b_only, i_only = rows[-1]
    cnt[b_only, i_only] = 0
    factor = {b: {} for b in range(B)}
    for (b, i) in rows:
        t = wl.t_first[b] + i
        factor[b][t] = 1e5
        factor[b][t - 1] = 1e-6
    for p in OL.window_of(wl, b_only, wl.t_first[b_only] + i_only):
        factor[b_only][int(p)] = 1e-6

    def latent(b, pos):
        f = torch.tensor([factor[b].get(int(p), 1.0) for p in pos], dtype=torch.float32)
        return wl.swa_latent(0, b, torch.as_tensor(pos)) * f[:, None]

    codes = g.swa_codes[0].clone()
    scales = g.swa_scales[0].clone()
    pos0 = wl.swa_pos0()
    for b in range(B):
        ts = [wl.t_first[b] + i for (bb, i) in rows if bb == b]
        if not ts:
            continue
        pos = np.unique(np.concatenate([OL.window_of(wl, b, t) for t in ts]))
        lat = latent(b, pos).to(dev).contiguous()
        c_dev = torch.empty(len(pos), d, dtype=torch.uint8, device=dev)
        s_dev = torch.empty(len(pos), dtype=torch.float32, device=dev)
        abi.csa2_pack_swa_fp8(lat, c_dev, s_dev)
        r = torch.as_tensor(pos - int(pos0[b]), device=dev)
        codes[b, r] = c_dev
        scales[b, r] = s_dev

    win = abi.Window(codes=codes.data_ptr(), scales=scales.data_ptr(), pos0=g.swa_pos0.data_ptr())
    O = torch.full_like(g.O[0], float("nan"))
    lse = torch.full_like(g.lse[0], float("nan"))
    tau = 1.0 / math.sqrt(d)
    abi.csa2_sparse_attn(g.dims(), g.cache(), win, Q, g.q_pos, g.idx[0], cnt, tau, O, lse)
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    ops = {}
    for (b, i) in rows:
        op = ops.setdefault(b, Operands(g, wl, b))   # the GPU's packed rows, verified first
        n = int(cnt[b, i])
        sel = g.idx[0][b, i, :n].cpu().numpy()
        wc, ws = F.fp8_pack(latent(b, OL.window_of(wl, b, wl.t_first[b] + i)).numpy())
        Qr = Q[b, i].cpu().double().numpy()
        kv, wv = op.kv_rows(sel), F.fp8_unpack_bf16(wc, ws)
        O_ref, lse_ref = A.sparse_attention(Qr, kv, wv, tau)
        Og = O[b, i].cpu().numpy()
        assert np.all(np.isfinite(Og)), (b, i)
        err = parity.attn_err(Og, O_ref)
        assert err <= parity.ATTN_RTOL, f"token {(b, i)}: attention error {err}"
        # logits reach ~1e5 here: the normaliser's log agrees within the fp32 accumulation
        # error of the logits, 2^-20 of the largest sum of |q_i k_i| * tau of each head
        keys = np.concatenate([kv, wv], axis=0)
        cond = (np.abs(Qr) @ np.abs(keys).T).max(axis=1) * tau
        lg = lse[b, i].cpu().double().numpy()
        tol = parity.LSE_ATOL + 2.0 ** -20 * cond
        assert np.all(np.abs(lg - lse_ref) <= tol), f"token {(b, i)}: lse {lg[:4]} vs {lse_ref[:4]}"
