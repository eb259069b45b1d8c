"""The C-ABI library loads without a GPU, exports every function include/attn46.h
declares, and rejects bad arguments before touching the device (CPU only)."""

import ctypes
import os
import re

import pytest

from exact_attention_46_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"attn_fwd", "attn_fwd_fp8", "hadamard_rotate_quant_fp8", "attn_check"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, n


def test_version(lib):
    assert lib.attn_version() == 120


FAKE = 1 << 20   # 16-byte aligned non-null fake device addresses: never dereferenced


@pytest.mark.parametrize("args,code", [
    ((None, FAKE, FAKE, FAKE * 4, None, 1, 1, 128, 128, 0, 0.0, 0), 1),
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 0, 128, 0, 0.0, 0), 1),      # S = 0
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 0, 1, 128, 128, 0, 0.0, 0), 1),    # B = 0
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 96, 0, 0.0, 0), 2),     # D = 96
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 0, 0, 0.0, 0), 1),      # D = 0
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 128, 2, 0.0, 0), 1),    # causal = 2
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 128, 0, -1.0, 0), 1),   # scale < 0
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 128, 0, float("nan"), 0), 1),
    ((FAKE + 8, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 128, 0, 0.0, 0), 1),  # misaligned
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 2, None, 1, 1, 128, 128, 0, 0.0, 0), 1),    # o aliases k
    ((FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 1, 128, 128, 0, 0.0, 7), 1),    # dtype
])
def test_attn_fwd_rejects_bad_arguments_without_launching(lib, args, code):
    assert lib.attn_fwd(*args, None) == code
    assert lib.attn_get_last_error()


def test_quantiser_and_fp8_reject_bad_arguments(lib):
    assert lib.hadamard_rotate_quant_fp8(None, FAKE, FAKE * 2, None, 1, 1, 128, 128, None) == 1
    assert lib.hadamard_rotate_quant_fp8(FAKE, FAKE * 8, FAKE * 16, None, 1, 1, 128, 48, None) == 2
    assert lib.hadamard_rotate_quant_fp8(FAKE, FAKE * 8, FAKE * 16, FAKE + 4, 1, 1, 128, 128, None) == 1
    assert lib.attn_fwd_fp8(FAKE, FAKE * 2, FAKE * 3, None, FAKE * 5, FAKE * 6, FAKE * 7, None,
                            1, 1, 128, 128, 0, 0.0, None) == 1
    assert lib.attn_selftest_bounded_wait(0, None) == 1


def test_rotary_entry_points_reject_bad_arguments(lib):
    f = lib.rope_hadamard_rotate_quant_fp8
    assert f(FAKE, None, 256, FAKE * 8, FAKE * 16, None, 1, 1, 128, 128, None) == 1      # no table
    assert f(FAKE, FAKE * 32, 127, FAKE * 8, FAKE * 16, None, 1, 1, 100, 128, None) == 1  # short table
    assert f(FAKE, FAKE * 32, 255, FAKE * 8, FAKE * 16, None, 1, 1, 129, 128, None) == 1  # needs 256 rows
    assert f(FAKE, FAKE * 32 + 8, 256, FAKE * 8, FAKE * 16, None, 1, 1, 128, 128, None) == 1  # misaligned
    assert f(FAKE, FAKE * 32, 256, FAKE * 8, FAKE * 16, None, 1, 1, 128, 96, None) == 2   # D = 96
    assert f(FAKE, FAKE * 8, 256, FAKE * 8, FAKE * 16, None, 1, 1, 128, 128, None) == 1   # out on table
    t = lib.rope_cos_sin_table
    assert t(None, 16, 128, 10000.0, None) == 1
    assert t(FAKE, 0, 128, 10000.0, None) == 1
    assert t(FAKE, 16, 63, 10000.0, None) == 1
    assert t(FAKE, 16, 128, 0.0, None) == 1
    assert t(FAKE, 16, 128, float("inf"), None) == 1
    assert t(FAKE + 4, 16, 128, 10000.0, None) == 1


def test_varlen_rejects_bad_arguments(lib):
    f = lib.attn_fwd_varlen
    ok = (FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, FAKE * 8, 2, 300, 200, 2, 128, 0, 0.0, None)
    def bad(i, val, code=1):
        a = list(ok)
        a[i] = val
        assert f(*a) == code, (i, val)
    bad(5, None)                  # no cu_seqlens
    bad(5, FAKE * 8 + 2)          # misaligned cu_seqlens
    bad(6, 0)                     # n_seq = 0
    bad(6, 4097)                  # too many sequences
    bad(7, 0)                     # total = 0
    bad(8, 0)                     # max_seqlen = 0
    bad(8, 262145, 2)             # max_seqlen above the level limit (D = 128)
    bad(10, 96, 2)                # D = 96
    bad(11, 3)                    # causal = 3
    bad(3, FAKE * 2)              # o aliases k
    bad(5, FAKE * 4)              # cu_seqlens inside o


def test_backward_rejects_bad_arguments(lib):
    f = lib.attn_bwd
    ws = lib.attn_bwd_workspace_bytes(1, 2, 300)
    assert ws == 8 * 2 * 384
    assert lib.attn_bwd_workspace_bytes(0, 2, 300) == 0
    ok = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 7, FAKE * 8, FAKE * 9, FAKE * 10, ws,
          1, 2, 300, 128, 0, 0.0, None]
    def bad(i, val, code=1):
        a = list(ok)
        a[i] = val
        assert f(*a) == code, (i, val)
    bad(5, None)                  # no lse
    bad(9, None)                  # no workspace
    bad(10, ws - 1)               # workspace too small
    bad(14, 256, 2)               # D = 256 unsupported here
    bad(14, 96, 2)                # D = 96
    bad(15, 2)                    # causal = 2
    bad(6, FAKE * 3)              # dq aliases v
    bad(9, FAKE * 8)              # workspace on dk
    bad(4, FAKE * 5 + 8)          # misaligned dout


def test_grouped_query_backward_rejects_bad_arguments(lib):
    f = lib.attn_bwd_gqa
    B, Hq, Hkv, S, D = 1, 8, 2, 300, 128
    ws = lib.attn_bwd_workspace_bytes(B, Hq, S)
    kv_bytes = 2 * B * S * Hkv * D        # 153,600: dk, dv sized by the key/value heads
    ok = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 7, FAKE * 8, FAKE * 9, FAKE * 10, ws,
          B, Hq, Hkv, S, D, 0, 0.0, None]
    def bad(i, val, code=1):
        a = list(ok)
        a[i] = val
        assert f(*a) == code, (i, val)
    bad(13, 3)                    # Hq not a multiple of Hkv
    bad(13, 0)                    # Hkv = 0
    bad(12, 0)                    # Hq = 0
    bad(13, 16)                   # Hkv > Hq
    bad(15, 256, 2)               # D = 256 unsupported here
    bad(10, lib.attn_bwd_workspace_bytes(B, Hkv, S))   # workspace sized by the wrong head count
    bad(7, FAKE * 2)              # dk aliases k
    bad(8, FAKE * 8 + kv_bytes - 16)   # dv overlaps the last row of dk
    bad(6, FAKE * 3 - 16)         # dq runs into v


def test_backward_without_workspace_rejects_problems_beyond_its_scratch(lib):
    # 2 * 16 * 65664 rows * 8 bytes > 16 MiB: rejected before any device work
    f = lib.attn_bwd_noalloc
    args = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 7, FAKE * 8, FAKE * 9,
            2, 16, 65537, 128, 0, 0.0, None]
    assert f(*args) == 1
    assert b"built-in scratch" in lib.attn_get_last_error()
    args[9] = 0
    assert f(*args) == 1


def test_gqa_and_decode_reject_bad_arguments(lib):
    g = lib.attn_fwd_gqa
    ok = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, 1, 8, 2, 256, 128, 0, 0.0, None]
    for i, val, code in ((6, 3, 1), (7, 0, 1), (9, 96, 2), (0, None, 1), (1, FAKE * 2 + 8, 1), (3, FAKE * 2, 1)):
        a = list(ok)
        a[i] = val
        assert g(*a) == code, (i, val)
    d = lib.attn_decode
    ok = [FAKE, FAKE * 8, FAKE * 16, FAKE * 24, None, None, 0, 1, 8, 2, 1, 4096, 128, 0, 0.0, None]
    for i, val, code in ((10, 5000, 1),      # Sq > Sk
                         (10, 33, 2),        # G * Sq = 4 * 33 > 128
                         (12, 256, 2),       # D = 256
                         (8, 6, 1)):         # Hq not a multiple of Hkv
        a = list(ok)
        a[i] = val
        assert d(*a) == code, (i, val)
    assert lib.attn_decode_workspace_bytes(0, 8, 2, 1, 4096, 128) == 0


def test_varlen_fp8_and_quantiser_reject_bad_arguments(lib):
    assert lib.attn_varlen_scale_blocks(300, 3) == 300 // 128 + 3 + 1
    assert lib.attn_varlen_scale_blocks(-1, 3) == 0
    q = lib.hadamard_rotate_quant_fp8_varlen
    ok = [FAKE, FAKE * 4, FAKE * 8, None, FAKE * 12, 3, 300, 2, 128, None]
    for i, val, code in ((4, None, 1),          # cu_seqlens missing
                         (4, FAKE * 12 + 2, 1), # misaligned
                         (5, 0, 1),             # n_seq = 0
                         (5, 5000, 1),          # n_seq above 4096
                         (8, 96, 2),            # D = 96
                         (1, FAKE, 1),          # out aliases x
                         (2, None, 1)):         # scale missing
        a = list(ok)
        a[i] = val
        assert q(*a) == code, (i, val)
    r = lib.rope_hadamard_rotate_quant_fp8_varlen
    ok = [FAKE, FAKE * 20, 256, FAKE * 4, FAKE * 8, None, FAKE * 12, 3, 300, 2, 128, None]
    for i, val, code in ((1, None, 1),          # rope_cs missing
                         (2, 100, 1),           # fewer than 128 table rows
                         (6, None, 1),          # cu_seqlens missing
                         (7, 0, 1),             # n_seq = 0
                         (10, 96, 2)):          # D = 96
        a = list(ok)
        a[i] = val
        assert r(*a) == code, (i, val)
    f = lib.attn_fwd_varlen_fp8
    ok = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 8, None, FAKE * 12, 3, 300, 200, 2, 128,
          0, 0.0, None]
    for i, val, code in ((3, None, 1),           # q_scale missing
                         (5, FAKE * 6 + 1, 1),   # v_scale misaligned
                         (8, None, 1),           # cu_seqlens missing
                         (9, 0, 1),              # n_seq = 0
                         (11, 0, 1),             # max_seqlen = 0
                         (13, 96, 2)):           # D = 96
        a = list(ok)
        a[i] = val
        assert f(*a) == code, (i, val)


def test_gqa_fp8_rejects_bad_arguments(lib):
    g = lib.attn_fwd_gqa_fp8
    ok = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 8, None, 1, 8, 2, 256, 128, 0, 0.0, None]
    for i, val, code in ((3, None, 1),            # q_scale missing
                         (5, FAKE * 6 + 1, 1),    # v_scale misaligned
                         (9, 3, 1),               # Hq not a multiple of Hkv
                         (10, 0, 1),              # Hkv = 0
                         (12, 96, 2),             # D = 96
                         (0, None, 1),            # q8 missing
                         (6, FAKE * 2, 1)):       # o aliases k8
        a = list(ok)
        a[i] = val
        assert g(*a) == code, (i, val)


def test_decode_fp8_rejects_bad_arguments(lib):
    d = lib.attn_decode_fp8
    ok = [FAKE, FAKE * 8, FAKE * 16, FAKE * 24, FAKE * 25, FAKE * 26, FAKE * 32, None, None, 0,
          1, 8, 2, 1, 4096, 128, 0, 0.0, None]
    for i, val, code in ((3, None, 1),           # q_scale missing
                         (5, None, 1),           # v_scale missing
                         (4, FAKE * 25 + 2, 1),  # k_scale misaligned
                         (13, 5000, 1),          # Sq > Sk
                         (13, 33, 2),            # G * Sq = 4 * 33 > 128
                         (15, 256, 2),           # D = 256
                         (15, 96, 2),            # D = 96
                         (11, 6, 1),             # Hq not a multiple of Hkv
                         (6, FAKE * 16, 1)):     # o aliases v
        a = list(ok)
        a[i] = val
        assert d(*a) == code, (i, val)


def test_missing_library_raises_instead_of_falling_back(monkeypatch, tmp_path):
    # with no compiled library every binding raises; nothing computes the result another way
    import torch
    from exact_attention_46_gb300 import ops
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    x = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ImportError):
        _lib.load()
    with pytest.raises((ImportError, ValueError)):
        ops.attn_fwd(x, x, x)
    with pytest.raises(ImportError):
        ops.varlen_scale_blocks(300, 3)


def _plan(lib, n_items, sms, key_tiles, max_parts):
    out = (ctypes.c_longlong * 3)()
    assert lib.attn_key_split_plan(n_items, sms, key_tiles, max_parts, out) == 0
    return tuple(out)


def test_key_split_plan_cases(lib):
    # B=2, S=8192, D=128 on 152 SMs (64 key tiles): 1024 blocks = 6 rounds + 112; four ranges
    # cost 3 rounds of (16 + 4) + 4 = 64 tiles against 68 unsplit: not worth it
    assert _plan(lib, 1024, 152, 64, 4) == (1024, 0, 1)
    # H = 17: 24 blocks left, one round of quarter ranges, 24 tiles against 68
    assert _plan(lib, 1088, 152, 64, 4) == (1064, 24, 4)
    assert _plan(lib, 1088, 152, 64, 2) == (1064, 24, 2)      # capped at two ranges: 40 tiles
    # H = 15: 48 left; thirds fit one round (30 tiles), quarters need two (44)
    assert _plan(lib, 960, 152, 64, 4) == (912, 48, 3)
    # B=1, S=32K (256 key tiles): 72 left, halves: 128 + 4 + 4 = 136 against 260
    assert _plan(lib, 2048, 152, 256, 4) == (1976, 72, 2)
    assert _plan(lib, 1216, 152, 64, 4) == (1216, 0, 1)       # whole rounds
    assert _plan(lib, 100, 152, 64, 4) == (100, 0, 1)         # no full round
    assert _plan(lib, 1088, 152, 64, 1) == (1088, 0, 1)       # split turned off
    # 12 key tiles: halves cost 14 of 16 (over 85 %), thirds 12; quarters would have 3 tiles
    assert _plan(lib, 176, 152, 12, 4) == (152, 24, 3)
    out = (ctypes.c_longlong * 3)()
    assert lib.attn_key_split_plan(10, 0, 4, 4, out) == 1
    assert lib.attn_key_split_plan(10, 152, 4, 4, None) == 1


def test_key_split_plan_is_the_cheapest_last_round(lib):
    # every plan: whole rounds first, the rest cut into ranges of >= 4 tiles; the chosen count
    # is the cheapest under the documented cost model and costs at most 85 % of no split
    for sms in (7, 152):
        for n_items in range(1, 3 * sms + 5, 3):
            for key_tiles in (1, 7, 8, 12, 16, 64, 256):
                for max_parts in (1, 2, 4, 9):
                    w, t, s = _plan(lib, n_items, sms, key_tiles, max_parts)
                    assert w + t == n_items
                    if n_items <= sms or n_items % sms == 0:
                        assert (t, s) == (0, 1)
                        continue
                    tail = n_items % sms
                    whole = key_tiles + 4
                    cost = {k: -(-tail * k // sms) * (-(-key_tiles // k) + 4) + 4
                            for k in range(2, min(max_parts, 4) + 1) if key_tiles >= 4 * k}
                    best = min(cost.values(), default=None)
                    if s == 1:
                        assert t == 0 and (best is None or 100 * best > 85 * whole)
                    else:
                        assert w % sms == 0 and t == tail and cost[s] == best <= 0.85 * whole
                        assert all(cost[k] > best for k in cost if k < s)


def test_split_forward_rejects_bad_arguments_without_a_gpu(lib):
    # dtype, scale-array combinations and the workspace are checked before any device call
    bad = [
        # bf16 with scales
        (FAKE, FAKE * 2, FAKE * 3, FAKE * 8, FAKE * 9, FAKE * 10, FAKE * 4, None, 1, 2, 2, 128, 128, 0, 0.0, 0),
        # E4M3 with only two of the three scale arrays
        (FAKE, FAKE * 2, FAKE * 3, FAKE * 8, None, FAKE * 10, FAKE * 4, None, 1, 2, 2, 128, 128, 0, 0.0, 1),
        # dtype out of range
        (FAKE, FAKE * 2, FAKE * 3, None, None, None, FAKE * 4, None, 1, 2, 2, 128, 128, 0, 0.0, 5),
        # Hq not a multiple of Hkv
        (FAKE, FAKE * 2, FAKE * 3, None, None, None, FAKE * 4, None, 1, 3, 2, 128, 128, 0, 0.0, 0),
    ]
    for a in bad:
        assert lib.attn_fwd_split(*a, None, 0, None) == 1, a
    # a misaligned or overlapping workspace
    base = (FAKE, FAKE * 2, FAKE * 3, None, None, None, FAKE * 4, None, 1, 2, 2, 128, 128, 0, 0.0, 0)
    assert lib.attn_fwd_split(*base, FAKE * 6 + 8, 4096, None) == 1
    assert lib.attn_fwd_split(*base, FAKE * 2, 4096, None) == 1


def test_split_workspace_bytes_of_invalid_shapes_is_zero(lib):
    for a in ((0, 16, 8192, 128, 0), (2, 16, 0, 128, 0), (2, 16, 8192, 96, 0), (2, 16, 8192, 128, 3)):
        assert lib.attn_fwd_split_workspace_bytes(*a) == 0
