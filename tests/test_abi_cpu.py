"""The C-ABI library loads, exports every declared symbol and validates arguments (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as m

    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    return sorted(set(re.findall(r"MSA_API[^;(]*?\b(msa_\w+)\s*\(", src, flags=re.S)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 7, names
    cdll = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(cdll, n), n
    assert set(lib.EXPORTED) == set(names)


def test_version(lib):
    assert lib.msa_version() >> 16 == 1


def test_workspace_sizes(lib):
    s = lib.Shape(B=1, T=1024, Hq=8, G=2, k=4)
    t = lib.msa_workspace_size(s, lib.MSA_WS_TOPK)
    f = lib.msa_workspace_size(s, lib.MSA_WS_FWD)
    b = lib.msa_workspace_size(s, lib.MSA_WS_BWD)
    assert 0 < t <= f <= b
    # fwd partial outputs dominate: k * hg * d bf16 per (b, t, g)
    assert f >= 1024 * 2 * 4 * 4 * 128 * 2
    assert lib.msa_workspace_size(s, 7) == 0


@pytest.mark.parametrize("kw", [dict(d=64), dict(d_idx=32), dict(Bk=64), dict(T=1000), dict(k=129),
                                dict(Hq=12, G=4), dict(Hq=7, G=2), dict(T=0), dict(B=0), dict(T=(1 << 20) + 128)])
def test_unsupported_shapes_have_no_workspace(lib, kw):
    base = dict(B=1, T=1024, Hq=8, G=2, k=4)
    base.update(kw)
    assert lib.msa_workspace_size(lib.Shape(**base), lib.MSA_WS_BWD) == 0


def test_validation_happens_before_any_device_work(lib):
    s = lib.Shape(B=1, T=1024, Hq=8, G=2, k=4)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_index_topk(s, 0, 0, 0, 0, stream=0, workspace_bytes=0)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG and "q_idx" in str(e.value)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_index_topk(s, 4096, 4096, 4096, 0, stream=0, workspace_bytes=0)
    assert e.value.status == lib.MSA_ERR_WORKSPACE
    with pytest.raises(lib.MsaError) as e:
        lib.msa_index_topk(s, 4096, 4096, 4096, 4096, stream=0, workspace_bytes=16)
    assert e.value.status == lib.MSA_ERR_WORKSPACE and "needed" in str(e.value)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_index_topk(s, 4097, 4096, 4096, 4096, stream=0, workspace_bytes=1 << 30)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG and "aligned" in str(e.value)
    bad = lib.Shape(B=1, T=1024, Hq=8, G=2, k=4, d=96)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_sparse_fwd(bad, 4096, 4096, 4096, 4096, 4096, 4096, 4096, stream=0, workspace_bytes=1 << 30)
    assert e.value.status == lib.MSA_ERR_UNSUPPORTED


def test_warmup_selection_validates_before_device_work(lib):
    # full attention needs every visible block: k >= T / Bk
    with pytest.raises(lib.MsaError) as e:
        lib.msa_warmup_block_idx(lib.Shape(B=1, T=1024, Hq=8, G=2, k=4), 4096, stream=0)
    assert e.value.status == lib.MSA_ERR_UNSUPPORTED and "k >= T / Bk" in str(e.value)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_warmup_block_idx(lib.Shape(B=1, T=1024, Hq=8, G=2, k=8), 0, stream=0)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG and "block_idx" in str(e.value)


def test_timing_events_validate_without_device(lib):
    with pytest.raises(lib.MsaError) as e:
        lib.msa_set_timing_events(5, None, None)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG
    with pytest.raises(lib.MsaError) as e:
        lib.msa_set_timing_events(lib.MSA_TIME_BWD, 4096, None)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG
    lib.msa_set_timing_events(lib.MSA_TIME_BWD, None, None)  # clearing is always fine


def test_selection_width_limits(lib):
    # the forward and backward take up to 128 blocks per row; the index top-k keeps at most 64
    s = lib.Shape(B=1, T=16384, Hq=8, G=2, k=128)
    assert lib.msa_workspace_size(s, lib.MSA_WS_BWD) > 0
    assert lib.msa_workspace_size(s, lib.MSA_WS_FWD) > 0
    assert lib.msa_workspace_size(s, lib.MSA_WS_TOPK) == 0
    assert lib.msa_workspace_size(s, lib.MSA_WS_TOPK_FP8) == 0
    assert lib.msa_workspace_size(lib.Shape(B=1, T=16384, Hq=8, G=2, k=64), lib.MSA_WS_TOPK) > 0
    with pytest.raises(lib.MsaError) as e:
        lib.msa_index_topk(s, 4096, 4096, 4096, 4096, stream=0, workspace_bytes=1 << 30)
    assert e.value.status == lib.MSA_ERR_UNSUPPORTED and "at most 64" in str(e.value)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_index_topk_fp8(s, 4096, 4096, 4096, 4096, stream=0, workspace_bytes=1 << 30)
    assert e.value.status == lib.MSA_ERR_UNSUPPORTED


def test_full_attention_shapes_and_validation(lib):
    # the full-attention calls take no block list: any k, heads per group 4 or 8, T up to 2^20
    for kw in (dict(k=1), dict(k=1024), dict(T=131072, k=16), dict(Hq=64, G=8)):
        base = dict(B=1, T=1024, Hq=8, G=2)
        base.update(kw)
        s = lib.Shape(**base)
        assert lib.msa_workspace_size(s, lib.MSA_WS_DENSE) >= 256 + s.B * s.T * (s.Hq + s.G) * 4
    for kw in (dict(Hq=4, G=2), dict(Hq=8, G=8), dict(d=64), dict(T=1000)):
        base = dict(B=1, T=1024, Hq=8, G=2, k=4)
        base.update(kw)
        assert lib.msa_workspace_size(lib.Shape(**base), lib.MSA_WS_DENSE) == 0
    s = lib.Shape(B=1, T=1024, Hq=8, G=2, k=1024)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_dense_fwd(s, 0, 4096, 4096, 4096, 4096, 4096, stream=0, workspace_bytes=1 << 20)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG and "Q" in str(e.value)
    with pytest.raises(lib.MsaError) as e:
        lib.msa_dense_fwd(lib.Shape(B=1, T=1024, Hq=4, G=2, k=1), 4096, 4096, 4096, 4096, 4096, 4096, stream=0,
                          workspace_bytes=1 << 20)
    assert e.value.status == lib.MSA_ERR_UNSUPPORTED and "heads per group" in str(e.value)
    args = [4096] * 8 + [1.0] + [4096] * 6  # Q .. k_idx, kl_weight, dQ .. KL
    with pytest.raises(lib.MsaError) as e:
        lib.msa_dense_bwd(s, *args, 4096, stream=0, workspace_bytes=16)
    assert e.value.status == lib.MSA_ERR_WORKSPACE
    with pytest.raises(lib.MsaError) as e:
        lib.msa_dense_bwd(s, *args[:8], float("nan"), *args[9:], 4096, stream=0, workspace_bytes=1 << 30)
    assert e.value.status == lib.MSA_ERR_INVALID_ARG and "kl_weight" in str(e.value)
