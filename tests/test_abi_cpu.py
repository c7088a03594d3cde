"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mla():
    from mla_absorbed_decode_gb300 import build_lib
    build_lib.build()
    import mla_absorbed_decode_gb300 as m
    m.lib()
    return m


def _declared():
    with open(os.path.join(ROOT, "include", "mla.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_exported(mla):
    names = _declared()
    assert len(names) >= 11
    handle = ctypes.CDLL(mla.library_path)
    for n in names:
        assert hasattr(handle, n), n
    assert set(names) == set(mla.EXPORTED_SYMBOLS)


def test_status_strings(mla):
    L = mla.lib()
    assert L.mla_status_string(0) == b"MLA_OK"
    assert L.mla_status_string(5) == b"MLA_ERR_TIMEOUT"
    assert L.mla_status_string(99) == b"MLA_ERR_UNKNOWN"


def test_sizes(mla):
    assert mla.metadata_size(64, 76) == (8 * 76 + 65) * 4
    assert mla.metadata_size(0, 0) == 0
    rows = 2 * 128
    ws = mla.decode_workspace_size(64, 2, 128, 38)
    assert ws >= (64 + 38) * rows * 513 * 4 and ws % 256 == 0
    assert mla.decode_workspace_size(0, 1, 1, 1) == 0
    fixed, hbm, split_cost = mla.schedule_params()
    assert fixed >= 0 and hbm >= 1 and split_cost >= 0


def test_host_argument_checks(mla):
    L = mla.lib()
    A = 0x10000  # a 16-byte aligned address that is never dereferenced on these paths
    ws = mla.decode_workspace_size(2, 1, 16, 4)
    # a valid-looking argument list; every case below breaks one argument, so the
    # call returns before touching the device (these addresses are never used)
    args = [A, A, 10, A, 8, A, 2, 1, 16, 0.1, 0, A, 4, A, ws, A, A, None]
    bad_null = list(args); bad_null[0] = None
    assert L.mla_decode(*bad_null) == 1                     # MLA_ERR_INVALID_ARG
    bad_align = list(args); bad_align[1] = A + 2
    assert L.mla_decode(*bad_align) == 1
    bad_shape = list(args); bad_shape[7] = 5; bad_shape[8] = 128   # s_q * H = 640 > 512
    assert L.mla_decode(*bad_shape) == 2                    # MLA_ERR_UNSUPPORTED
    small_ws = list(args); small_ws[14] = ws - 1
    assert L.mla_decode(*small_ws) == 3                     # MLA_ERR_WORKSPACE
    nan_scale = list(args); nan_scale[9] = float("nan")
    assert L.mla_decode(*nan_scale) == 1
    for bad in (0.0, -0.5):   # the kernel takes the row maximum on unscaled scores
        neg_scale = list(args); neg_scale[9] = bad
        assert L.mla_decode(*neg_scale) == 1
    # the FP8 entry: the same checks, plus its scale
    f8 = args[:2] + [1.0] + args[2:]
    assert L.mla_decode_fp8(*f8[:1], None, *f8[2:]) == 1      # no cache
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        bad_kv = list(f8); bad_kv[2] = bad
        assert L.mla_decode_fp8(*bad_kv) == 1
    bad_shape8 = list(f8); bad_shape8[8] = 5; bad_shape8[9] = 128
    assert L.mla_decode_fp8(*bad_shape8) == 2
    small_ws8 = list(f8); small_ws8[15] = ws - 1
    assert L.mla_decode_fp8(*small_ws8) == 3
    # the sparse FP8 entry: a list is required, the scale must be finite and positive, and
    # the sparse decode's own checks apply
    # (q, kv, scale, num_blocks, table, max_blocks, seqlens, indices, stride, topk_lens, B, s_q, H,
    #  softmax_scale, causal, metadata, parts, workspace, bytes, out, lse, stream)
    sp8 = [A, A, 1.0, 10, A, 8, A, A, 8, A, 2, 1, 16, 0.1, 0, A, 4, A, ws, A, A, None]
    no_list = list(sp8); no_list[7] = None
    assert L.mla_decode_sparse_fp8(*no_list) == 1
    for bad in (0.0, -2.0, float("nan")):
        bad_kv = list(sp8); bad_kv[2] = bad
        assert L.mla_decode_sparse_fp8(*bad_kv) == 1
    bad_stride = list(sp8); bad_stride[8] = 0
    assert L.mla_decode_sparse_fp8(*bad_stride) == 1
    bad_rows = list(sp8); bad_rows[11] = 5; bad_rows[12] = 128
    assert L.mla_decode_sparse_fp8(*bad_rows) == 2
    assert L.mla_decode_metadata(None, 2, 1, 16, 0, 4, A, None) == 1
    assert L.mla_decode_metadata(A, 2, 8, 128, 0, 4, A, None) == 2
    assert L.mla_decode_metadata(A, 16385, 1, 128, 0, 4, A, None) == 2   # more requests than supported
    assert L.mla_absorb_q(A, 100, None, 0, A, A, 4, 1, None) == 1      # stride below H*128
    assert L.mla_absorb_q(A, 128, A, 8, A, A, 4, 1, None) == 1         # q_pe stride below H*64
    assert L.mla_unabsorb_o(A + 8, A, A, 4, 1, None) == 1
    assert L.mla_num_sm_parts(0, 5, 128) < 0


def test_fp8_projection_argument_checks(mla):
    L = mla.lib()
    A = 0x10000  # 16-byte aligned, never dereferenced: every case returns before any launch
    ws = mla.bmm_fp8_workspace_size()
    assert ws >= 4 * 128
    # (q_nope, stride, q_pe, pe_stride, positions, theta, w_uk_t, w_scale, q, N, H, workspace, bytes, stream)
    ab = [A, 128, A, 64, A, 10000.0, A, 2.0 ** -9, A, 4, 1, A, ws, None]
    for i in (0, 6, 8):                                             # q_nope, weights, q
        bad = list(ab); bad[i] = None
        assert L.mla_absorb_q_fp8(*bad) == 1                        # MLA_ERR_INVALID_ARG
    for bad_scale in (0.0, -1.0, float("nan"), float("inf")):
        bad = list(ab); bad[7] = bad_scale
        assert L.mla_absorb_q_fp8(*bad) == 1
    bad = list(ab); bad[1] = 100                                    # stride below H*128
    assert L.mla_absorb_q_fp8(*bad) == 1
    bad = list(ab); bad[2] = None                                   # positions without q_pe
    assert L.mla_absorb_q_fp8(*bad) == 1
    bad = list(ab); bad[5] = 1.0                                    # rope_theta must exceed 1
    assert L.mla_absorb_q_fp8(*bad) == 1
    bad = list(ab); bad[12] = ws - 1
    assert L.mla_absorb_q_fp8(*bad) == 3                            # MLA_ERR_WORKSPACE
    bad = list(ab); bad[11] = None
    assert L.mla_absorb_q_fp8(*bad) == 3
    # (o_lat, w_uv_t, w_scale, o, N, H, workspace, bytes, stream)
    un = [A, A, 2.0 ** -9, A, 4, 1, A, ws, None]
    assert L.mla_unabsorb_o_fp8(*([A + 8] + un[1:])) == 1            # misaligned o_lat
    bad = list(un); bad[2] = 0.0
    assert L.mla_unabsorb_o_fp8(*bad) == 1
    bad = list(un); bad[7] = 0
    assert L.mla_unabsorb_o_fp8(*bad) == 3


def test_absorb_plan_argument_checks(mla):
    L = mla.lib()
    A = 0x10000  # 16-byte aligned, never dereferenced: every case returns before any launch
    assert L.mla_absorb_plan_max_batch() >= 1024
    # (q_nope, stride, q_pe, pe_stride, positions, theta, w_uk, q, N, H, seqlens, B, parts, metadata, stream)
    ok = [A, 128, A, 64, A, 10000.0, A, A, 8, 1, A, 4, 76, A, None]
    for i in (0, 6, 7, 10, 13):                                     # q_nope, w_uk, q, seqlens, metadata
        bad = list(ok); bad[i] = None
        assert L.mla_absorb_q_plan(*bad) == 1                       # MLA_ERR_INVALID_ARG
    for i, v in ((11, 0), (11, 3), (12, 0), (8, 0), (9, 0)):        # B < 1, N not a multiple of B, parts, N, H
        bad = list(ok); bad[i] = v
        assert L.mla_absorb_q_plan(*bad) == 1
    bad = list(ok); bad[13] = A + 2                                 # metadata must be 4-byte aligned
    assert L.mla_absorb_q_plan(*bad) == 1
    bad = list(ok); bad[2] = None                                   # positions without q_pe
    assert L.mla_absorb_q_plan(*bad) == 1
    bad = list(ok); bad[5] = 1.0                                    # rope_theta must exceed 1
    assert L.mla_absorb_q_plan(*bad) == 1
    big = L.mla_absorb_plan_max_batch() + 1
    bad = list(ok); bad[11] = big; bad[8] = big                     # more requests than the CTA's shared memory holds
    assert L.mla_absorb_q_plan(*bad) == 2                           # MLA_ERR_UNSUPPORTED
    bad = list(ok); bad[9] = 1024; bad[8] = 4                       # s_q * H beyond a cluster's pairs
    assert L.mla_absorb_q_plan(*bad) == 2


def test_absorb_fp8_plan_argument_checks(mla):
    L = mla.lib()
    A = 0x10000  # 16-byte aligned, never dereferenced: every case returns before any launch
    ws = mla.bmm_fp8_workspace_size()
    # (q_nope, stride, q_pe, pe_stride, positions, theta, w_uk_t, w_scale, q, N, H, workspace, bytes,
    #  seqlens, B, parts, metadata, stream)
    ok = [A, 128, A, 64, A, 10000.0, A, 2.0 ** -9, A, 8, 1, A, ws, A, 4, 76, A, None]
    for i in (13, 16):                                              # seqlens, metadata
        bad = list(ok); bad[i] = None
        assert L.mla_absorb_q_fp8_plan(*bad) == 1                   # MLA_ERR_INVALID_ARG
    for i, v in ((14, 0), (14, 3), (15, 0)):                        # B < 1, N not a multiple of B, parts
        bad = list(ok); bad[i] = v
        assert L.mla_absorb_q_fp8_plan(*bad) == 1
    bad = list(ok); bad[2] = None                                   # positions without q_pe
    assert L.mla_absorb_q_fp8_plan(*bad) == 1
    big = L.mla_absorb_plan_max_batch() + 1
    bad = list(ok); bad[14] = big; bad[9] = big
    assert L.mla_absorb_q_fp8_plan(*bad) == 2                       # MLA_ERR_UNSUPPORTED
    for i in (0, 6, 8):                                             # q_nope, weights, q (checked by the FP8 bmm)
        bad = list(ok); bad[i] = None
        assert L.mla_absorb_q_fp8_plan(*bad) == 1
    bad = list(ok); bad[12] = ws - 1
    assert L.mla_absorb_q_fp8_plan(*bad) == 3                       # MLA_ERR_WORKSPACE
