"""Host-side checks of the C ABI that need no GPU: the library loads on a
machine without a driver, exports every symbol include/msa.h declares, and
rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import block_sparse_attention_proxy_gb300 as m

    if not os.path.exists(m.LIB_PATH):
        from block_sparse_attention_proxy_gb300 import build

        build.build()
    m.load()
    return m


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", src)))


def test_exports_match_header(m):
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    assert sorted(m.EXPORTS) == declared
    lib = m.load()
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(m):
    for code in range(7):
        assert m.msa_status_string(code).startswith(m._abi.STATUS_NAMES[code])


def test_workspace_sizes_and_shape_checks(m):
    ok = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4)
    assert m.msa_select_workspace_size(ok) > 0
    assert m.msa_fwd_workspace_size(ok) > m.msa_select_workspace_size(ok)
    assert m.msa_bwd_workspace_size(ok) > 0
    for bad in (m.make_params(1024, 1, 1024, 4, 1, 96, 32, 4),   # d
                m.make_params(1024, 1, 1024, 4, 1, 64, 48, 4),   # dp
                m.make_params(1024, 1, 1024, 12, 4, 64, 32, 4),  # G = 3
                m.make_params(1024, 1, 1024, 4, 1, 64, 32, 17),  # top_k
                m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, block=64),
                m.make_params(1024, 1, 1024, 4, 3, 64, 32, 4),   # hq % hkv
                m.make_params(1024, 1, 2048, 4, 1, 64, 32, 4),   # max_seqlen > T
                m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, softmax_scale=0.0),
                m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, flags=2)):  # unknown flag bit
        assert m.msa_fwd_workspace_size(bad) == 0
    reuse = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, flags=m.MSA_FLAG_REUSE_REGROUP)
    assert m.msa_bwd_workspace_size(reuse) == m.msa_bwd_workspace_size(ok)
    stall = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, flags=m.MSA_FLAG_TEST_STALL_SELECT)
    assert m.msa_select_workspace_size(stall) == m.msa_select_workspace_size(ok)
    both = m.MSA_FLAG_TEST_STALL_SELECT | m.MSA_FLAG_REUSE_REGROUP | 0x200  # one unknown bit
    assert m.msa_select_workspace_size(m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4,
                                                     flags=both)) == 0


def _call_fwd(m, prm, ptr_val, ws_bytes):
    lib = m.load()
    p = ctypes.c_void_p(ptr_val)
    return lib.msa_fwd(ctypes.byref(prm), p, p, p, p, p, p, p, p, p, p, ws_bytes, None)


def test_host_errors_before_any_launch(m):
    prm = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4)
    need = m.msa_fwd_workspace_size(prm)
    lib = m.load()
    assert _call_fwd(m, prm, 0, need) == 1                 # null pointers
    assert _call_fwd(m, prm, 0x1008, need) == 1            # misaligned (8 bytes)
    assert _call_fwd(m, prm, 0x1000, need - 1) == 3        # workspace too small
    bad = m.make_params(1024, 1, 1024, 4, 1, 96, 32, 4)
    assert _call_fwd(m, bad, 0x1000, need) == 2            # unsupported d
    assert lib.msa_set_profile_events(7, None, None) == 1
    # an empty batch is a no-op that returns OK without touching the GPU
    empty = m.make_params(0, 1, 0, 4, 1, 64, 32, 4)
    assert _call_fwd(m, empty, 0x1000, 0) == 0


def test_params_layout_matches_header(m):
    # 11 int32, 3 float, 1 uint32, in the header's order
    assert ctypes.sizeof(m.MsaParams) == 15 * 4
    names = [f[0] for f in m.MsaParams._fields_]
    assert names == ["total_tokens", "num_docs", "max_seqlen", "hq", "hkv", "d", "dp", "block",
                     "top_k", "window", "dilation", "softmax_scale", "proxy_scale", "kl_weight",
                     "flags"]
    assert m.MsaParams.window.offset == 9 * 4 and m.MsaParams.flags.offset == 14 * 4


def test_block_pattern_params_checked_on_host(m):
    ok = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, window=3, dilation=2)
    assert m.msa_fwd_workspace_size(ok) > 0
    zero_dil = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, window=2, dilation=0)
    assert m.msa_fwd_workspace_size(zero_dil) == m.msa_fwd_workspace_size(ok)  # 0 reads as 1
    for bad in (dict(window=4), dict(window=-1), dict(window=1, dilation=-2)):
        assert m.msa_select_workspace_size(m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4, **bad)) == 0


def test_launch_counter_starts_at_zero_without_gpu(m):
    if torch.cuda.is_available():
        pytest.skip("counter may have advanced in this process")
    assert m.msa_launch_count() == 0


def test_host_input_step_needs_one_buffer_set(m):
    """The host-input step rotates `depth` sets of device buffers; fewer than
    one is rejected before any device memory is touched."""
    from block_sparse_attention_proxy_gb300.step import HostInputStep

    prm = m.make_params(1024, 1, 1024, 4, 1, 64, 32, 4)
    for depth in (0, -1):
        with pytest.raises(ValueError):
            HostInputStep(prm, {}, device="cpu", depth=depth)
