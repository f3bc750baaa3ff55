"""The C-ABI library: it builds, loads without a GPU, exports every symbol
include/fa.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import exact_attention_79_gb300 as fa
    if not os.path.exists(fa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return fa.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    import exact_attention_79_gb300 as fa
    names = declared_functions()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), n
        assert n in fa.SIGNATURES, n


def test_status_strings_and_version(lib):
    for code in range(8):
        assert lib.fa_status_string(code)
    assert lib.fa_version() >= 100


def test_ex2_probe_rejects_a_null_result_pointer(lib):
    assert lib.fa_ex2_throughput(None, None) == 1


def test_workspace_size_formula(lib):
    # lse2 + D: B*Hq*ceil(N/128)*128 floats each; dQ accumulator: B*Hq*N*d floats
    assert lib.fa_bwd_workspace_bytes(1, 16, 16, 8192, 128) == 2 * 16 * 8192 * 4 + 16 * 8192 * 128 * 4
    # B*Hq = 8 rows of ceil(100/128)*128 = 128 padded entries: 4096 B each for lse2 and D
    assert lib.fa_bwd_workspace_bytes(2, 4, 2, 100, 64) == 4096 + 4096 + 8 * 100 * 64 * 4
    assert lib.fa_bwd_workspace_bytes(1, 3, 2, 128, 128) == 0      # Hq not a multiple of Hkv
    assert lib.fa_bwd_workspace_bytes(1, 2, 2, 128, 100) == 0      # head dim not a multiple of 8
    # above d = 128 the three-pass backward keeps no dQ accumulator: lse2 + D only
    assert lib.fa_bwd_workspace_bytes(1, 2, 2, 128, 136) == 2 * 2 * 128 * 4


def test_invalid_arguments_rejected_without_device(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    assert lib.fa_fwd(null, fake, fake, fake, fake, 1, 1, 1, 128, 64, 0, 0.125, null) == 1
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 128, 84, 0, 0.125, null) == 1     # d not a multiple of 8
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 4, 3, 128, 64, 0, 0.125, null) == 1
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 128, 64, 0, 0.0, null) == 1
    assert lib.fa_fwd(fake, fake, fake, fake, ctypes.c_void_p((1 << 20) + 4), 1, 1, 1, 128, 64, 0, 0.1, null) == 1
    assert lib.fa_fwd_f32(fake, fake, fake, fake, fake, 1, 1, 1, 128, 128, 0, 0.1, null) == 2
    args = [fake] * 9
    assert lib.fa_bwd(*args, null, 1 << 30, 1, 1, 1, 128, 128, 1, 0.1, null) == 6
    assert lib.fa_bwd(*([null] + [fake] * 8), fake, 1 << 30, 1, 1, 1, 128, 128, 1, 0.1, null) == 1


def test_head_dim_and_fp8_rules_without_device(lib):
    """Head dims 8..256 for the forward and for fa_bwd, fa_bwd_kv,
    fa_bwd_deterministic and fa_bwd_noalloc, 8..128 for the single backward
    phases and the block-sparse backward, multiples of 16 up to 256 for FP8:
    the host checks answer before any device work."""
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 128, 264, 0, 0.125, null) == 1    # past 256
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 128, 252, 0, 0.125, null) == 1    # not a multiple of 8
    args = [fake] * 9
    # backward above 128: the three-pass path, which checks its workspace first
    assert lib.fa_bwd(*args, null, 0, 1, 1, 1, 128, 256, 1, 0.1, null) == 6
    assert lib.fa_bwd_deterministic(*args, null, 0, 1, 1, 1, 128, 192, 1, 0.1, null) == 6
    assert lib.fa_bwd_kv(*args, null, 0, 1, 1, 1, 128, 300, 200, 1, 0.1, null) == 6
    assert lib.fa_bwd_workspace_bytes(1, 2, 2, 128, 256) == 2 * 2 * 128 * 4
    # beyond the no-alloc scratch (32 MiB of LSE and D: 4 M rows) at d = 256
    assert lib.fa_bwd_noalloc(*args, 1, 64, 64, 65536 + 128, 256, 1, 0.1, null) == 6
    # the single phases and the block-sparse backward stop at 128
    assert lib.fa_bwd_blocksparse_workspace_bytes(1, 2, 2, 128, 192) == 0
    assert lib.fa_bwd_preprocess(fake, fake, fake, fake, 1 << 30, 1, 1, 1, 128, 136, null) == 2
    assert lib.fa_bwd_dkdv(*([fake] * 7), 1 << 30, 1, 1, 1, 128, 256, 1, 0.1, null) == 2
    # FP8: multiples of 16 up to 256; other multiples of 8 are valid arguments
    # but not built (a row of codes must be a multiple of 16 bytes for TMA)
    assert lib.fa_fwd_fp8(*([fake] * 8), 1, 1, 1, 128, 8, 0, 0.1, null) == 2
    assert lib.fa_fwd_fp8_kv(*([fake] * 8), 1, 1, 1, 128, 300, 152, 0, 0.1, null) == 2
    assert lib.fa_fwd_fp8(*([fake] * 8), 1, 1, 1, 128, 264, 0, 0.1, null) == 1
    assert lib.fa_fp8_quantize_v(fake, fake, fake, 4, 100, 200, null) == 2
    assert lib.fa_fwd_fp8(*([fake] * 7 + [null]), 1, 1, 1, 128, 128, 0, 0.1, null) == 1
    assert lib.fa_fp8_quantize_rows(fake, fake, fake, 4, 100, 40, null) == 2
    assert lib.fa_fp8_quantize_v(fake, fake, fake, 0, 100, 128, null) == 1
    # scale-array and padded-key helpers
    assert lib.fa_fp8_row_scales(1) == 1 and lib.fa_fp8_row_scales(64) == 1 and lib.fa_fp8_row_scales(65) == 2
    assert lib.fa_fp8_vt_keys(1) == 128 and lib.fa_fp8_vt_keys(128) == 128 and lib.fa_fp8_vt_keys(129) == 256
    assert lib.fa_fp8_row_scales(0) == 0 and lib.fa_fp8_vt_keys(0) == 0


def test_binding_refuses_mismatched_tensors_before_any_launch(lib):
    """Shapes and dtypes are checked for every tensor before placement, so CPU
    tensors show it: a wrong output, gradient, workspace or FP8 scale buffer
    never reaches a kernel that would write or read past its end."""
    import torch
    import exact_attention_79_gb300 as fa
    bf = torch.bfloat16
    q = torch.zeros(1, 2, 64, 64, dtype=bf)
    k = torch.zeros(1, 1, 64, 64, dtype=bf)
    lse = torch.zeros(1, 2, 64)
    with pytest.raises(ValueError, match="^v:"):
        fa.fwd(q, k, torch.zeros(1, 1, 64, 32, dtype=bf))
    with pytest.raises(ValueError, match="^out:"):
        fa.fwd(q, k, k, out=torch.zeros(1, 2, 64, 64))
    with pytest.raises(ValueError, match="^lse:"):
        fa.fwd(q, k, k, lse=torch.zeros(1, 2, 63))
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.fwd(q, k, k)
    with pytest.raises(ValueError, match="^do:"):
        fa.bwd(q, k, k, q, lse, torch.zeros(1, 2, 64, 32, dtype=bf))
    with pytest.raises(ValueError, match="^dk:"):
        fa.bwd(q, k, k, q, lse, q, workspace=torch.zeros(16, dtype=torch.uint8), dk=torch.zeros(1, 2, 64, 64, dtype=bf))
    with pytest.raises(ValueError, match="^workspace:"):
        fa.bwd(q, k, k, q, lse, q, workspace=torch.zeros(16, dtype=torch.float32))
    u8 = torch.uint8
    q8, k8 = torch.zeros(1, 2, 64, 64, dtype=u8), torch.zeros(1, 1, 64, 64, dtype=u8)
    qs, ks = torch.zeros(1, 2, 1), torch.zeros(1, 1, 1)
    vt8, vs = torch.zeros(1, 1, 64, 128, dtype=u8), torch.zeros(1, 1, 64)
    with pytest.raises(ValueError, match="^v_scale:"):
        fa.fwd_fp8(q8, qs, k8, ks, vt8, torch.zeros(1, 1, 64, dtype=bf))
    with pytest.raises(ValueError, match="^vt8:"):
        fa.fwd_fp8(q8, qs, k8, ks, torch.zeros(1, 1, 64, 64, dtype=u8), vs)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.fwd_fp8(q8, qs, k8, ks, vt8, vs)
    with pytest.raises(ValueError, match="^v:"):
        fa.quantize_fp8(q, k, torch.zeros(1, 1, 64, 64))
