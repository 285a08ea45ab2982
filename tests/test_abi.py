"""Host-side checks of the C-ABI library (no GPU needed): it loads, it exports
every symbol include/dg_canvas.h declares, and host validation rejects bad
arguments with the documented codes before any kernel could launch."""
import ctypes
import os
import re

import pytest

from canvas_denoising_gb300 import binding as B
from canvas_denoising_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^DG_API\s+[\w\s\*]+?\b(dg_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(B.EXPORTS), names ^ set(B.EXPORTS)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = B.status_string(code)
        assert s.startswith("DG_")
    assert B.status_string(12345) == "unknown dg_status"


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first


def test_renoise_rejects_bad_arguments(lib):
    assert lib.dg_renoise(None, FAKE, FAKE, 16, 512, 0.5, 0, 0, 0, None, None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_renoise(FAKE, FAKE, FAKE, 0, 512, 0.5, 0, 0, 0, None, None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_renoise(FAKE, FAKE, FAKE, 16, 0, 0.5, 0, 0, 0, None, None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_renoise(FAKE, FAKE, FAKE, 16, 512, float("nan"), 0, 0, 0, None, None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_canvas_init(None, 16, 512, 0, 0, None) == B.DG_ERR_INVALID_ARG


def test_kv_append_rejects_overflow_and_leaves_len(lib):
    n = ctypes.c_int64(100)
    rc = lib.dg_kv_append(FAKE, FAKE, 120, ctypes.byref(n), FAKE, FAKE, 32, 2, 128, B.DG_BF16, None, 0, None, None,
                          None, 0, None)
    assert rc == B.DG_ERR_INVALID_ARG and n.value == 100
    rc = lib.dg_kv_append(FAKE, FAKE, 1000, ctypes.byref(n), FAKE, FAKE, 32, 2, 96, B.DG_BF16, None, 0, None, None,
                          None, 0, None)
    assert rc == B.DG_ERR_UNSUPPORTED and n.value == 100
    misaligned = ctypes.c_void_p((1 << 20) + 8)
    rc = lib.dg_kv_append(misaligned, FAKE, 1000, ctypes.byref(n), FAKE, FAKE, 32, 2, 128, B.DG_BF16, None, 0, None,
                          None, None, 0, None)
    assert rc == B.DG_ERR_INVALID_ARG and n.value == 100


def test_attn_rejects_bad_arguments(lib):
    args = [FAKE, FAKE, FAKE, 4352, 4096, FAKE, FAKE, FAKE, None, 256, 16, 8, 128, -1.0, B.DG_BF16, 0, None, 0, None]
    a = list(args); a[11] = 5  # Hq % Hkv != 0
    assert lib.dg_canvas_attn(*a) == B.DG_ERR_INVALID_ARG
    a = list(args); a[12] = 80
    assert lib.dg_canvas_attn(*a) == B.DG_ERR_UNSUPPORTED
    a = list(args); a[4] = 5000  # prefix beyond capacity
    assert lib.dg_canvas_attn(*a) == B.DG_ERR_INVALID_ARG
    a = list(args); a[15] = 7
    assert lib.dg_canvas_attn(*a) == B.DG_ERR_INVALID_ARG
    need = lib.dg_canvas_attn_workspace_size(256, 16, 8, 128, 4096, B.DG_BF16)
    assert need > 0
    assert lib.dg_canvas_attn(*args) == B.DG_ERR_WORKSPACE


def test_vocab_step_rejects_bad_arguments(lib):
    need = lib.dg_vocab_step_workspace_size(256, 262144, 2816, B.DG_BF16)
    assert need > 262144 * 256 * 2  # the bf16 P ring is part of it
    base = [FAKE, FAKE, 256, 262144, 2816, B.DG_BF16, FAKE, FAKE, FAKE, FAKE, FAKE, need, None]
    a = list(base); a[4] = 2800  # d % 64
    assert lib.dg_vocab_step(*a) == B.DG_ERR_UNSUPPORTED
    a = list(base); a[2] = 300
    assert lib.dg_vocab_step(*a) == B.DG_ERR_UNSUPPORTED
    a = list(base); a[11] = need - 1
    assert lib.dg_vocab_step(*a) == B.DG_ERR_WORKSPACE
    a = list(base); a[0] = None
    assert lib.dg_vocab_step(*a) == B.DG_ERR_INVALID_ARG
    a = list(base); a[10] = ctypes.c_void_p((1 << 20) + 16)  # workspace not 256-byte aligned
    assert lib.dg_vocab_step(*a) == B.DG_ERR_INVALID_ARG
    a = list(base); a[5] = 7
    assert lib.dg_vocab_step(*a) == B.DG_ERR_INVALID_ARG


def test_vocab_plan_is_a_host_query(lib):
    import ctypes
    buf = (ctypes.c_int32 * 6)()
    assert lib.dg_vocab_step_plan(256, 262144, 2816, B.DG_BF16, ctypes.cast(buf, ctypes.c_void_p)) == B.DG_OK
    n_a, n_c, ks, pair, grid, n_vt = list(buf)
    assert n_vt == 1024 and n_a + n_c == grid
    if pair:
        # CTA pairs: consumers own 256-column slices, 2816 = 11 of them per residue class
        assert n_a % 2 == 0 and n_c == 2 * 11 * ks and grid <= 152
    else:
        assert n_c % 11 == 0 and n_c // 11 == ks
    assert lib.dg_vocab_step_plan(256, 262144, 2800, B.DG_BF16, ctypes.cast(buf, ctypes.c_void_p)) == B.DG_ERR_INVALID_ARG


@pytest.mark.parametrize("C,V,d", [
    (256, 262144, 2816), (256, 32768, 1024), (256, 65536, 2816), (1, 1, 64), (77, 33333, 192), (200, 9000, 320),
    (256, 100, 4160), (256, 2000, 8192), (256, 262144, 8192), (130, 7000, 768), (256, 20000, 640), (256, 257, 64),
])
def test_vocab_plans_are_consistent(lib, C, V, d):
    """For shapes across the supported range: both roles present, the grid
    fits the GPU (152 SMs without a device), CTA pairs come in twos, the
    residue classes do not outnumber the tiles, and the workspace holds at
    least the P ring and the consumers' fp32 partials."""
    plan = B.vocab_step_plan(C, V, d)
    n_vt = (V + 255) // 256
    assert plan["vocab_tiles"] == n_vt
    assert plan["producers"] >= 1 and plan["consumers"] >= 1
    assert plan["producers"] + plan["consumers"] == plan["ctas"] <= 152
    assert 1 <= plan["vocab_split"] <= n_vt
    if plan["cluster_pairs"]:
        assert plan["producers"] % 2 == 0 and plan["consumers"] % 2 == 0
        assert plan["producers"] // 2 <= n_vt
    ring = n_vt * 256 * 256 * 2                 # bf16 P for every row and vocabulary id
    partials = plan["vocab_split"] * 256 * d * 4
    assert B.vocab_step_workspace_size(C, V, d) >= ring + partials


def test_debug_inject_validates(lib):
    assert lib.dg_debug_inject(7, 0) == B.DG_ERR_INVALID_ARG
    assert lib.dg_debug_inject(1, -1) == B.DG_ERR_INVALID_ARG
    assert lib.dg_debug_inject(1, 20000) == B.DG_ERR_INVALID_ARG
    assert lib.dg_debug_inject(0, 0) == B.DG_OK  # clearing needs no device
