"""The C-ABI library loads and exports every entry point of include/csa2.h; host
validation rejects bad arguments before any launch (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from compressed_sparse_attention_05_gb300 import abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def _declared():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(csa2_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(abi.SIGNATURES) == names


def test_abi_version(lib):
    assert abi.csa2_abi_version() == 2


FAKE = 1 << 20  # an aligned non-null address; validation fails before any use


def _err(rc):
    return rc, lib_err()


def lib_err():
    return abi.lib().csa2_last_error().decode()


def test_pack_validation(lib):
    assert lib.csa2_pack_mxfp4_f32(FAKE, 4, 15, FAKE, FAKE, None) == 1
    assert "multiple of 16" in lib_err()
    assert lib.csa2_pack_mxfp4_f32(None, 4, 16, FAKE, FAKE, None) == 1
    assert "x must not be NULL" in lib_err()
    assert lib.csa2_pack_mxfp4_f32(FAKE + 4, 4, 16, FAKE, FAKE, None) == 1
    assert "aligned" in lib_err()
    assert lib.csa2_pack_mxfp4_f32(None, 0, 16, None, None, None) == 0   # empty: nothing to do
    assert lib.csa2_pack_swa_fp8(FAKE, -1, 16, FAKE, FAKE, None) == 1


def _dims(**kw):
    d = dict(B=2, Tq=1, d=512, r=64, Hq=64, Hi=8, Di=128, idx_dtype=abi.CSA2_BF16, K=512, W=128,
             max_pages=4, n_pool_blocks=2048, pool_block=8, swa_cap=128)
    d.update(kw)
    return abi.Dims(**d)


def _cache():
    return abi.Cache(kv_codes=FAKE, kv_scales=FAKE, idx_k=FAKE, page_table=FAKE, n_entries=FAKE, n_pages=8)


def test_index_topk_validation(lib):
    dm, c = _dims(), _cache()
    need = abi.csa2_index_topk_workspace_size(dm, 256)
    assert need > 2 * 2048 * 8 * 4
    call = lambda dims, ws, nbytes: lib.csa2_index_topk(  # noqa: E731
        C.byref(dims), C.byref(c), FAKE, FAKE, FAKE, None, None, FAKE, FAKE, None, None, 256, ws, nbytes, None)
    assert call(dm, FAKE, need - 1) == 4
    assert "workspace" in lib_err()
    assert call(_dims(K=4096), FAKE, need) == 1
    assert call(_dims(Di=48), FAKE, need) == 1
    assert call(_dims(Hi=17), FAKE, need) == 1


def test_attention_validation(lib):
    c, w = _cache(), abi.Window(codes=FAKE, scales=FAKE, pos0=FAKE)
    call = lambda dims, O: lib.csa2_sparse_attn(  # noqa: E731
        C.byref(dims), C.byref(c), C.byref(w), FAKE, FAKE, FAKE, FAKE, 0.1, O, None, None)
    assert call(_dims(d=256), FAKE) == 2                  # unsupported width
    assert call(_dims(), None) == 1
    assert "O must not be NULL" in lib_err()
    assert call(_dims(B=0), None) == 0                    # empty batch: no launch


def test_layer_validation(lib):
    a = abi.LayerArgs()
    a.mode = 7
    assert lib.csa2_layer(C.byref(a), None, 0, None) == 1
    assert "unknown mode" in lib_err()
    a.mode = abi.MODE_REINDEX
    a.dims = _dims()
    a.cache = _cache()
    a.q_pos = a.idx_out = a.cnt_out = FAKE
    assert lib.csa2_layer(C.byref(a), None, 0, None) == 1   # REINDEX without a pool
    assert "pool" in lib_err()


def test_compress_validation(lib):
    dm, c = _dims(), _cache()
    rc = lib.csa2_compress_pack(FAKE, 2, 64, 100, FAKE, FAKE, 1e-6, 1e4, None, FAKE, C.byref(dm), C.byref(c),
                                FAKE, 1 << 30, None)
    assert rc == 1 and "multiple of 64" in lib_err()
    need = abi.csa2_compress_workspace_size(2, 64, 128, 512, 128)
    rc = lib.csa2_compress_pack(FAKE, 2, 64, 128, FAKE, FAKE, 1e-6, 1e4, FAKE, FAKE, C.byref(dm), C.byref(c),
                                FAKE, need - 1, None)
    assert rc == 4


def test_compress_layers_validation(lib):
    dm, c = _dims(), _cache()
    caches = (abi.Cache * 2)(c, c)
    rc = lib.csa2_compress_layers(FAKE, 2, 64, 128, 0, FAKE, 128, FAKE, 1e-6, 1e4, FAKE, C.byref(dm), caches,
                                  FAKE, 1 << 30, None)
    assert rc == 1 and "L must be" in lib_err()
    rc = lib.csa2_compress_layers(FAKE, 2, 64, 128, 2, FAKE, 96, FAKE, 1e-6, 1e4, FAKE, C.byref(dm), caches,
                                  FAKE, 1 << 30, None)
    assert rc == 1 and "Di must be" in lib_err()
    # grouped: one workspace for all layers' outputs, larger than one layer's
    one = abi.csa2_compress_workspace_size(2, 64, 128, 512, 128)
    assert abi.csa2_compress_layers_workspace_size(2, 64, 128, 2, 512, 128) > one
    need = abi.csa2_compress_layers_workspace_size(2, 64, 128, 2, 512, dm.Di)
    rc = lib.csa2_compress_layers(FAKE, 2, 64, 128, 2, FAKE, dm.Di, FAKE, 1e-6, 1e4, FAKE, C.byref(dm), caches,
                                  FAKE, need - 1, None)
    assert rc == 4


def test_swa_replay_validation(lib):
    win = abi.Window(codes=FAKE, scales=FAKE, pos0=FAKE)
    call = lambda dims, H, n_tok, nbytes: lib.csa2_swa_replay(  # noqa: E731
        FAKE, 2, n_tok, H, FAKE, FAKE, 1e-6, 1e4, FAKE, C.byref(dims), C.byref(win), FAKE, nbytes, None)
    assert call(_dims(), 100, 128, 1 << 30) == 1 and "multiple of 64" in lib_err()
    assert call(_dims(d=128), 128, 128, 1 << 30) == 2
    assert call(_dims(swa_cap=0), 128, 128, 1 << 30) == 1 and "swa_cap" in lib_err()
    assert call(_dims(B=3), 128, 128, 1 << 30) == 1 and "dims.B" in lib_err()
    assert call(_dims(), 128, 0, 0) == 0          # nothing to replay: no launch, no workspace
    need = abi.csa2_swa_replay_workspace_size(2, 128, 128, 512)
    assert need > 0 and need % (2 * 128 * 512 * 4) == 0   # whole split-K partial planes
    assert call(_dims(), 128, 128, need - 1) == 4
    assert lib.csa2_swa_replay(FAKE, 2, 128, 128, FAKE, FAKE, 1e-6, 1e4, FAKE, C.byref(_dims()), None, FAKE,
                               need, None) == 1 and "window" in lib_err()
