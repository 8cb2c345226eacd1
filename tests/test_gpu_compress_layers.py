"""Several layers' compression from one hidden state (csa2_compress_layers):
"DeepSeek-V4.1 架构解析" §01, every decoder layer projects its KV from the
last encoder layer's hidden state with its own weights.  Each layer's packed
entries and indexer keys against the oracle's compression of that layer."""
import numpy as np
import pytest
import torch

import parity
from compressed_sparse_attention_05_gb300 import abi, build
from oracle import compress as Cm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()


def _np(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("d,r,Di,idx_dtype,kv,G,L", [(512, 64, 128, "bf16", "mxfp4", 70, 3),
                                                    (512, 64, 0, "bf16", "mxfp4", 70, 3),
                                                    (64, 16, 32, "f32", "mxfp4", 70, 3),
                                                    (512, 64, 128, "bf16", "fp8", 70, 3),
                                                    (512, 64, 128, "bf16", "mxfp4", 256, 3),
                                                    (512, 64, 128, "bf16", "mxfp4", 507, 3),
                                                    (512, 64, 0, "bf16", "mxfp4", 507, 3),
                                                    (512, 64, 128, "bf16", "mxfp4", 70, 66)])
def test_compress_layers_matches_oracle(d, r, Di, idx_dtype, kv, G, L):
    """kv = "fp8": the V4-style main KV (E4M3 row + fp32 scale per entry).  G entries
    per sequence: 70 (one M tile), 256 (two: CTA pairs share each weight tile) and
    507 (four, the last ragged: clusters of four share it, the index-key tile's
    rows copied by two of them).  L = 66 layers: the per-layer packs run 64 layers
    per launch, so the last two go in a second launch."""
    fp8 = kv == "fp8"
    dev = "cuda"
    g = torch.Generator().manual_seed(21)
    B, H = 2, 256
    T = 4 * G + 1                         # G entries per sequence; the last token makes none
    assert T // 4 == G
    first = [10, 0]                       # entries before the new tokens
    eps, base = 1e-6, 10000.0
    hidden = torch.randn(B, T, H, generator=g).to(torch.bfloat16)
    W_all = (torch.randn(L, d + Di, 4 * H, generator=g) * 0.02).to(torch.bfloat16)
    gamma = 1.0 + 0.05 * torch.randn(L, d, generator=g)
    idx_t = torch.bfloat16 if idx_dtype == "bf16" else torch.float32
    pages = (max(first) + G + 63) // 64
    n_pages = B * pages
    caches, keep = [], []
    for l in range(L):
        perm = torch.randperm(n_pages, generator=g).to(torch.int32).reshape(B, pages)
        t = {"codes": torch.zeros(n_pages * 64, d if fp8 else d // 2, dtype=torch.uint8, device=dev),
             "scales": (torch.zeros(n_pages * 64, dtype=torch.float32, device=dev) if fp8
                        else torch.zeros(n_pages * 64, d // 16, dtype=torch.uint8, device=dev)),
             "idx": torch.zeros(n_pages * 64, max(Di, 1), dtype=idx_t, device=dev),
             "pt": perm.to(dev), "n": torch.tensor([f + G for f in first], dtype=torch.int32, device=dev)}
        keep.append(t)
        caches.append(abi.Cache(kv_codes=t["codes"].data_ptr(), kv_scales=t["scales"].data_ptr(),
                                idx_k=t["idx"].data_ptr(), page_table=t["pt"].data_ptr(),
                                n_entries=t["n"].data_ptr(), n_pages=n_pages))
    dims = abi.Dims(B=B, Tq=T, d=d, r=r, Hq=4, Hi=4, Di=Di if Di else 32,
                    idx_dtype=abi.CSA2_BF16 if idx_dtype == "bf16" else abi.CSA2_F32, K=16, W=16,
                    max_pages=pages, n_pool_blocks=0, pool_block=8, swa_cap=0,
                    kv_format=abi.CSA2_KV_FP8 if fp8 else abi.CSA2_KV_MXFP4)
    ws = torch.empty(max(256, abi.csa2_compress_layers_workspace_size(B, T, H, L, d, Di)), dtype=torch.uint8,
                     device=dev)
    fe = torch.tensor(first, dtype=torch.int32, device=dev)
    abi.csa2_compress_layers(hidden.to(dev), W_all.to(dev), Di, gamma.to(dev), eps, base, fe, dims, caches, ws)
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    for l in range(L):
        W = _np(W_all[l, :d])
        Wi = _np(W_all[l, d:]) if Di else None
        for b in range(B):
            ref = Cm.compress_pack(_np(hidden[b]), W, _np(gamma[l]), eps, r, base, first[b], W_idx=Wi,
                                   idx_dtype=idx_dtype, kv_format=kv)
            ids = torch.from_numpy(ref["entry_ids"])
            assert len(ids) == G
            slots = keep[l]["pt"][b, ids // 64].long().cpu() * 64 + ids % 64
            codes = keep[l]["codes"][slots.to(dev)].cpu().numpy()
            scales = keep[l]["scales"][slots.to(dev)].cpu().numpy()
            # decided from the GEMM's fp32 sums: equal except one-step flips at rounding boundaries
            cat = Cm.concat_groups(_np(hidden[b]))
            tau_x = parity.latent_error_bound(ref["c"], parity.gemm_error_bound(cat, W), _np(gamma[l]), eps, r,
                                              ref["x"])
            if fp8:
                parity.check_fp8_after_gemm(codes, scales, ref["x"], tau_x)
            else:
                parity.check_mxfp4_after_gemm(codes, scales, ref["x"], tau_x)
            if Di:
                kk = keep[l]["idx"][slots.to(dev)].float().cpu().double().numpy()
                parity.check_keys_after_gemm(kk, cat @ Wi.T, parity.gemm_error_bound(cat, Wi), idx_dtype)
