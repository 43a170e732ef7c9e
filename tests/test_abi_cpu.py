"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from weight_only_quantized_qgemv_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


@pytest.fixture(scope="module")
def L():
    _build.build()          # nvcc cross-compiles sm_103a without a GPU
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(q\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["qgemv", "qgate_up", "qexpert_group", "qexpert_group_workspace", "qdequant", "qstatus_string",
              "qlast_cuda_error"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/qgemv.h but not exported"
        ctypes.cast(getattr(L, name), ctypes.c_void_p)


def test_status_strings(L):
    for st in range(0, -11, -1):
        assert _lib.qstatus_string(st) and "unknown status" not in _lib.qstatus_string(st)
    assert "unknown" in _lib.qstatus_string(-100)


# Fake but 256-byte aligned device addresses: the checks below fail before any
# pointer is used.
A = 1 << 20


@pytest.mark.parametrize("fmt,gs,I,want", [
    (3, 32, 1024, -1),          # unknown format
    (6, 0, 1024, -1),           # unknown format
    (2, 32, 1024, -1),          # int4 per row: gs must be 0 or I
    (2, 0, 1040, -2),           # int4 per row: I not a multiple of 32
    (13, 8, 1024, -1),          # int8 grouped: group below 16
    (13, 48, 1024, -1),         # int8 grouped: group not a power of two
    (13, 0, 1024, -1),          # int8 grouped: a group size is required
    (13, 1024, 2048, -1),       # int8 grouped: group above 512
    (13, 64, 1040, -2),         # int8 grouped: I not a multiple of gs
    (8, 64, 1024, -1),          # MXFP4 with ue8m0 bytes is group 32 only
    (8, 0, 1056, -2),           # ue8m0 bytes: I not a multiple of 128
    (4, 48, 1024, -1),          # int4 group size not a power of two
    (4, 16, 1024, -1),          # int4 group below 32
    (5, 32, 1024, -1),          # int3 is group 64 only
    (7, 64, 1024, -1),          # MXFP4 is group 32 only
    (1, 32, 1024, -1),          # int8 per row: gs must be 0 or I
    (1, 0, 1000, -2),           # int8 row not a multiple of 16
    (4, 64, 1056, -2),          # I not a multiple of gs
    (5, 0, 1000, -2),           # int3 I not a multiple of 64
    (4, 32, 51232, -2),         # row longer than the staging limit
    (4, 2048, 4096, -1),        # int4 group above 1024
])
def test_qgemv_rejects_bad_formats_and_sizes(L, fmt, gs, I, want):
    assert L.qgemv(fmt, gs, A, A, A, 16, I, 1, A, None) == want


def test_qgemv_rejects_null_and_misaligned(L):
    assert L.qgemv(4, 32, None, A, A, 16, 1024, 1, A, None) == -4
    assert L.qgemv(4, 32, A, A, None, 16, 1024, 1, A, None) == -4
    assert L.qgemv(4, 32, A + 8, A, A, 16, 1024, 1, A, None) == -3     # weights need 16 B
    assert L.qgemv(4, 32, A, A, A + 4, 16, 1024, 1, A, None) == -3     # x needs 16 B
    assert L.qgemv(4, 32, A, A + 2, A, 16, 1024, 1, A, None) == -3     # scales need 4 B
    assert L.qgemv(4, 32, A, A, A, 0, 1024, 1, A, None) == -2          # O >= 1
    assert L.qgemv(4, 32, A, A, A, 16, 1024, 0, A, None) == -2         # s >= 1


def test_qgate_up_and_dequant_checks(L):
    assert L.qgate_up(4, 32, A, A, A, A, A, 16, 1000, 1, A, None) == -2
    assert L.qgate_up(4, 32, A, A, None, A, A, 16, 1024, 1, A, None) == -4
    assert L.qdequant(9, 32, A, A, 16, 1024, A, None) == -1
    assert L.qdequant(4, 32, A, A, 16, 1024, None, None) == -4


def test_expert_group_checks(L):
    ws = _lib.qexpert_group_workspace(256, 6144, 2048, 8, 8)
    assert ws >= 64 * (6144 + 2048) * 4
    args = [4, 32, A, A, A, A, A, A, 256, 6144, 2048, A, 8, 8, A, A, A, A, ws, None, None]
    bad = list(args)
    bad[18] = ws - 1
    assert L.qexpert_group(*bad) == -5                 # workspace too small
    bad = list(args)
    bad[17] = A + 16
    assert L.qexpert_group(*bad) == -3                 # workspace must be 256-byte aligned
    bad = list(args)
    bad[12], bad[13] = 1024, 8                         # s * k above 4096
    assert L.qexpert_group(*bad) == -2
    bad = list(args)
    bad[10] = 2050                                     # F not a multiple of the group
    assert L.qexpert_group(*bad) == -2
    assert _lib.qexpert_group_workspace(0, 6144, 2048, 8, 8) >= 0


def test_activation_checks(L):
    """Unknown activations and limits that are negative or NaN are refused before any launch."""
    gu = lambda act, lim: L.qgate_up_act(4, 32, A, A, A, A, A, 16, 1024, 1, act, lim, A, None)
    assert gu(2, 1.0) == -9
    assert gu(1, -0.5) == -9
    assert gu(1, float("nan")) == -9
    assert gu(1, -0.5) == L.qgate_up_act(4, 32, A, A, A, A, A, 16, 1024, 1, 1, -0.5, A, None)
    # a bad activation is reported before a bad size
    assert L.qgate_up_act(4, 32, A, A, A, A, A, 16, 1000, 1, 3, 1.0, A, None) == -9
    ws = _lib.qexpert_group_workspace(256, 6144, 2048, 8, 8)
    args = [4, 32, A, A, A, A, A, A, 256, 6144, 2048, A, 8, 8, A, A, 1, float("nan"), A, A, ws, None, None]
    assert L.qexpert_group_act(*args) == -9
    args[16], args[17] = 7, 1.0
    assert L.qexpert_group_act(*args) == -9


def test_kernel_policy_round_trip(L):
    """The kernel-choice knob is host state only: set, read back, reject unknown values."""
    prev = _lib.qkernel_policy(_lib.QKERNEL_TILE)
    try:
        assert _lib.qkernel_policy(_lib.QKERNEL_RING) == _lib.QKERNEL_TILE
        assert L.qkernel_policy(7) == -1            # QSTATUS_BAD_FMT, policy unchanged
        assert _lib.qkernel_policy(_lib.QKERNEL_AUTO) == _lib.QKERNEL_RING
    finally:
        _lib.qkernel_policy(prev)


def test_qgemm_checks(L):
    """The prefill GEMM's host-side checks (nothing is enqueued)."""
    Z = ctypes.c_size_t
    L.qgemm.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p, ctypes.c_void_p, Z, ctypes.c_void_p]
    L.qgemm_workspace.argtypes = [ctypes.c_int, ctypes.c_int]
    L.qgemm_workspace.restype = Z
    ws = L.qgemm_workspace(6144, 512)
    assert ws >= 2 * 512 * 6144 * 2 + 512 * 4
    assert L.qgemm_workspace(6144, 20) == L.qgemm_workspace(6144, 32)     # rows padded to a 32-row tile
    assert L.qgemm_workspace(0, 4) == 0
    assert L.qgemm(4, 32, A, A, A, 16, 6176, 512, A, A, ws, None) == -2     # I not a multiple of 64
    assert L.qgemm(13, 16, A, A, A, 16, 1024, 64, A, A, ws, None) == -1     # partials need 32 inputs
    assert L.qgemm(3, 0, A, A, A, 16, 1024, 64, A, A, ws, None) == -1       # unknown format
    assert L.qgemm(4, 32, A, A, A, 16, 6144, 512, A, A, ws - 1, None) == -5  # workspace too small
    assert L.qgemm(4, 32, A, A, A, 16, 6144, 512, A, None, ws, None) == -4   # no workspace
    assert L.qgemm(4, 32, A, A, A, 16, 6144, 512, A, A + 16, ws, None) == -3  # workspace not 256-aligned
    assert L.qgemm(4, 32, A, A, A, 16, 6144, 0, A, A, ws, None) == -2       # s < 1
    assert L.qgemm(4, 32, A, A, A, 0, 6144, 512, A, A, ws, None) == -2      # O < 1
    big = L.qgemm_workspace((1 << 20) + 64, 1 << 17)
    assert L.qgemm(4, 32, A, A, A, 16, (1 << 20) + 64, 8, A, A, big, None) == -2   # I past 2^20
    assert L.qgemm(4, 32, A, A, A, 16, 64, (1 << 16) + 1, A, A, big, None) == -2   # s past 65536


def test_route_checks(L):
    """qroute / qexpert_group_routed host-side checks (nothing is enqueued)."""
    f = ctypes.c_float
    L.qroute.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 4 + \
        [f, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert L.qroute(2, A, A, 4, 256, 8, 1, 1.0, A, A, None) == -10            # unknown kind
    assert L.qroute(0, A, A, 4, 256, 8, 1, float("nan"), A, A, None) == -10   # NaN scale
    assert L.qroute(0, A, None, 4, 256, 33, 1, 1.0, A, A, None) == -2         # k above 32
    assert L.qroute(0, A, None, 4, 8, 9, 1, 1.0, A, A, None) == -2            # k above E
    assert L.qroute(0, A, None, 4, 1025, 8, 1, 1.0, A, A, None) == -2         # E above 1024
    assert L.qroute(0, A, None, 0, 256, 8, 1, 1.0, A, A, None) == -2          # no tokens
    assert L.qroute(1, A, None, 4, 256, 8, 1, 1.0, A, A, None) == -4          # sigmoid router needs a bias
    assert L.qroute(0, A + 2, None, 4, 256, 8, 1, 1.0, A, A, None) == -3      # misaligned logits
    Z = ctypes.c_size_t
    L.qexpert_group_routed.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 6 + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
         f, ctypes.c_int, f, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, Z, ctypes.c_void_p,
         ctypes.c_void_p]
    ws = _lib.lib().qexpert_group_workspace(256, 6144, 2048, 8, 8)
    base = [7, 0, A, A, A, A, A, A, 256, 6144, 2048, A, 8, 8]
    assert L.qexpert_group_routed(*base, 2, A, None, 1, 1.0, 0, 0.0, A, A, A, A, ws, None, None) == -10
    assert L.qexpert_group_routed(*base, 0, A, None, 1, 1.0, 5, 0.0, A, A, A, A, ws, None, None) == -9
    assert L.qexpert_group_routed(*base, 0, A, None, 1, 1.0, 0, 0.0, A, A, A, A, ws - 1, None, None) == -5
    # more experts than the fused routing holds (the router kernel would run
    # first): the expert group's checks still come before anything is enqueued
    # (with no device, an enqueued router would have returned QSTATUS_LAUNCH)
    ws512 = _lib.lib().qexpert_group_workspace(512, 6144, 2048, 8, 8)
    big = [7, 0, A + 8, A, A, A, A, A, 512, 6144, 2048, A, 8, 8]          # gate not 16-byte aligned
    assert L.qexpert_group_routed(*big, 0, A, None, 1, 1.0, 0, 0.0, A, A, A, A, ws512, None, None) == -3
    big = [7, 0, A, A, A, A, A, A, 512, 6144, 2048, A, 8, 8]
    assert L.qexpert_group_routed(*big, 0, A, None, 1, 1.0, 0, 0.0, A, A, A, A, ws512 - 1, None, None) == -5
    assert L.qexpert_group_routed(*big, 0, A, None, 1, 1.0, 0, 0.0, A, None, A, A, ws512, None, None) == -4
    assert L.qexpert_group_routed(*big, 0, A, None, 1, 1.0, 3, 0.0, A, A, A, A, ws512, None, None) == -9


def test_debug_inject_checks(L):
    """The test hook's arguments: unknown kinds and waits below 1 ns are refused; disarming always works."""
    assert L.qdebug_inject(5, 1000) == -2
    assert L.qdebug_inject(1, 0) == -2
    assert L.qdebug_inject(0, 0) == 0
    assert L.qdebug_inject(1, 1000000) == 0      # armed ...
    assert L.qdebug_inject(0, 0) == 0            # ... and disarmed again (no launch happens here)


def test_empty_sizes_are_rejected(L):
    """Zero rows, inputs or activation rows: QSTATUS_BAD_DIM before anything is enqueued."""
    assert L.qgemv(4, 32, A, A, A, 0, 1024, 1, A, None) == -2
    assert L.qgemv(4, 32, A, A, A, 16, 1024, 0, A, None) == -2
    assert L.qgemv(1, 0, A, A, A, 16, 0, 1, A, None) == -2
    assert L.qdequant(4, 32, A, A, 0, 1024, A, None) == -2


def test_binding_refuses_host_and_strided_tensors():
    """The binding passes device addresses only: a host tensor or a strided
    view is refused before the library is called."""
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib._ptr(torch.zeros(4))
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib._ptr(object())
    assert _lib._ptr(None) is None
    assert _lib._ptr(4096) == 4096

    class View:                         # a CUDA tensor's interface, strided
        is_cuda = True

        def is_contiguous(self):
            return False

        def data_ptr(self):
            raise AssertionError("must not be reached")
    with pytest.raises(ValueError, match="contiguous"):
        _lib._ptr(View())


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "qgemv.h"

static int fails = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("FAIL %s\n", #cond); fails++; } } while (0)

int main(void)
{
    int st;
    for (st = 0; st >= -10; st--) printf("%d %s\n", st, qstatus_string(st));
    EXPECT(strcmp(qstatus_string(12345), "unknown status") == 0);
    EXPECT(qgemm_workspace(6144, 512) > 0 && qgemm_workspace(0, 4) == 0);
    EXPECT(qexpert_group_workspace(256, 6144, 2048, 8, 8) > 0);
    /* host-side checks only: nothing reaches a device */
    EXPECT(qgemv(3, 0, NULL, NULL, NULL, 16, 1024, 1, NULL, NULL) == QSTATUS_BAD_FMT);
    EXPECT(qgemv(QFMT_INT4_G, 32, NULL, NULL, NULL, 16, 1024, 0, NULL, NULL) == QSTATUS_BAD_DIM);
    EXPECT(qgemv(QFMT_INT4_G, 32, NULL, NULL, NULL, 16, 1024, 1, NULL, NULL) == QSTATUS_NULL);
    EXPECT(qgemm(QFMT_INT3_G64, 0, NULL, NULL, NULL, 16, 1000, 4, NULL, NULL, 0, NULL) == QSTATUS_BAD_DIM);
    EXPECT(qroute(2, NULL, NULL, 1, 8, 2, 1, 1.0f, NULL, NULL, NULL) == QSTATUS_BAD_ROUTE);
    EXPECT(qgate_up_act(QFMT_MXFP4_G32, 0, NULL, NULL, NULL, NULL, NULL, 16, 64, 1, 7, 0.0f, NULL, NULL)
           == QSTATUS_BAD_ACT);
    EXPECT(qkernel_policy(99) == QSTATUS_BAD_FMT);
    EXPECT(qkernel_policy(QKERNEL_AUTO) == QKERNEL_AUTO);
    printf("fails %d\n", fails);
    return fails != 0;
}
"""


def test_header_compiles_as_c_and_cpp_and_links(L, tmp_path):
    """A plain C99 program, built with -Wall -Wextra -pedantic -Werror against
    include/qgemv.h and linked to the library, calls the entry points that need
    no GPU; the header also compiles as C++ (its extern "C" guard)."""
    import shutil
    import subprocess
    gcc, gxx = shutil.which("gcc"), shutil.which("g++")
    if not gcc or not gxx:
        pytest.skip("no host C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    libdir = os.path.dirname(_build.LIB)
    exe = tmp_path / "client"
    inc = os.path.join(ROOT, "include")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src), "-o", str(exe),
                    "-L", libdir, "-l:" + os.path.basename(_build.LIB), "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    cpp = tmp_path / "client.cpp"
    cpp.write_text('#include "qgemv.h"\nint main() { return qgemm_workspace(0, 0) != 0; }\n')
    subprocess.run([gxx, "-std=c++17", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", inc,
                    str(cpp)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.splitlines()
    assert lines[-1] == "fails 0"
    for line in lines[:11]:
        st, text = line.split(" ", 1)
        assert text == L.qstatus_string(int(st)).decode()


# The header's rules for format, group size and sizes, restated per format:
# (allowed gs values as a predicate of (gs, I), the multiple I must be).
_POW2 = lambda g, lo, hi: lo <= g <= hi and g & (g - 1) == 0
HEADER_RULES = {
    1: (lambda g, I: g in (0, I), lambda g: 16),                     # int8 per row
    2: (lambda g, I: g in (0, I), lambda g: 32),                     # int4 per row
    4: (lambda g, I: _POW2(g, 32, 1024), lambda g: g),               # int4 grouped
    5: (lambda g, I: g in (0, 64), lambda g: 64),                    # int3-g64
    7: (lambda g, I: g in (0, 32), lambda g: 32),                    # MXFP4, f32 scales
    8: (lambda g, I: g in (0, 32), lambda g: 128),                   # MXFP4, ue8m0 bytes
    13: (lambda g, I: _POW2(g, 16, 512), lambda g: g),               # int8 grouped
}


def expected_statuses(fmt, gs, I, dims_ok, gemm=False):
    """Every status the header allows for these arguments (NULL pointers):
    the statuses of all violated rules, or QSTATUS_NULL if none is violated."""
    bad = set()
    rule = HEADER_RULES.get(fmt)
    if rule is None or not rule[0](gs, I):
        bad.add(-1)
    else:
        if I % rule[1](gs):
            bad.add(-2)
        if gemm and (I if fmt in (1, 2) else {5: 64, 7: 32, 8: 32}.get(fmt, gs)) < 32:
            bad.add(-1)                                               # qgemm: groups of >= 32 inputs
    if not dims_ok:
        bad.add(-2)
    return bad or {-4}


def _draw_case(rng, i_max):
    fmt = int(rng.choice([1, 2, 4, 5, 7, 8, 13])) if rng.random() < 0.8 else int(rng.choice([0, 3, 6, -1, 99]))
    base = int(rng.choice([16, 32, 64, 128, 256, 1024]))
    I = int(rng.choice([base * int(rng.integers(1, max(2, i_max // base))), int(rng.integers(-64, 40000)), 0,
                        i_max, i_max + 64], p=[0.6, 0.25, 0.05, 0.05, 0.05]))
    likely = {1: [0, I], 2: [0, I], 4: [32, 64, 128, 256, 512, 1024], 5: [0, 64], 7: [0, 32], 8: [0, 32],
              13: [16, 32, 64, 128, 256, 512]}.get(fmt, [0])
    gs = int(rng.choice(likely)) if rng.random() < 0.6 else \
        int(rng.choice([0, 8, 16, 32, 48, 64, 128, 256, 512, 1024, 2048, I]))
    O = int(rng.choice([-1, 0, 1, int(rng.integers(1, 100000))]))
    s = int(rng.choice([-1, 0, 1, 8, 9, int(rng.integers(1, 70000))]))
    return fmt, gs, I, O, s


def test_size_checks_follow_the_header_rules(L):
    """qgemv, qdequant and qgemm on random formats, group sizes and sizes, all
    with NULL pointers (nothing reaches a device): the status is one the
    header's rules give for the violated rule, or QSTATUS_NULL when every size
    rule holds."""
    import numpy as np
    from collections import Counter
    seen = {"qgemv": Counter(), "qdequant": Counter(), "qgemm": Counter()}
    rng = np.random.default_rng(2024)
    Z = ctypes.c_size_t
    L.qgemm.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p, ctypes.c_void_p, Z, ctypes.c_void_p]
    for _ in range(3000):
        fmt, gs, I, O, s = _draw_case(rng, 36864)
        want = expected_statuses(fmt, gs, I, O >= 1 and 1 <= I <= 36864 and s >= 1)
        if 36864 < I <= 51200 and want == {-2}:
            # rows the header gives only as "about 37,000" at most: the
            # shared-memory budget is checked with the launch shape, after
            # the pointers
            want = {-2, -4}
        got = L.qgemv(fmt, gs, None, None, None, O, I, s, None, None)
        assert got in want, (fmt, gs, I, O, s, got, want)
        seen["qgemv"][got] += 1
        want = expected_statuses(fmt, gs, I, O >= 1 and I >= 1)
        got = L.qdequant(fmt, gs, None, None, O, I, None, None)
        assert got in want, ("qdequant", fmt, gs, I, O, got, want)
        seen["qdequant"][got] += 1
    for _ in range(3000):
        fmt, gs, I, O, s = _draw_case(rng, 1 << 20)
        dims_ok = O >= 1 and 1 <= I <= (1 << 20) and I % 64 == 0 and 1 <= s <= (1 << 16)
        want = expected_statuses(fmt, gs, I, dims_ok, gemm=True)
        got = L.qgemm(fmt, gs, None, None, None, O, I, s, None, None, 0, None)
        assert got in want, ("qgemm", fmt, gs, I, O, s, got, want)
        seen["qgemm"][got] += 1
    for name, c in seen.items():           # every outcome is reached often
        assert min(c[-1], c[-2], c[-4]) >= 100, (name, dict(c))


def test_expert_group_checks_follow_the_header_rules(L):
    """qexpert_group_act on random formats, group sizes, sizes, pair counts and
    activations, all with NULL pointers: the status is one the header's rules
    give for a violated rule (gs applies to the D-long gate/up rows and the
    F-long down rows alike; s * k <= 4096), or QSTATUS_NULL."""
    import math
    from collections import Counter

    import numpy as np
    rng = np.random.default_rng(2025)
    f = ctypes.c_float
    L.qexpert_group_act.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 6 + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, f,
         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    seen = Counter()
    for _ in range(4000):
        fmt, gs, D, _, s = _draw_case(rng, 36864)
        F = int(rng.choice([D, 2048, 128, 96, 40000, 0], p=[0.5, 0.2, 0.1, 0.1, 0.05, 0.05]))
        E = int(rng.choice([0, 1, 256, -3], p=[0.05, 0.2, 0.7, 0.05]))
        k = int(rng.choice([0, 1, 8, 32, 600], p=[0.05, 0.3, 0.4, 0.15, 0.1]))
        act = int(rng.choice([0, 1, 2, -1], p=[0.45, 0.45, 0.05, 0.05]))
        limit = float(rng.choice([0.0, 7.0, -1.0, math.inf, math.nan], p=[0.25, 0.45, 0.1, 0.1, 0.1]))
        want = set()
        if act not in (0, 1) or (act == 1 and not limit >= 0):
            want.add(-9)
        for n in (D, F):               # every violated rule of either row length
            if fmt not in HEADER_RULES or not HEADER_RULES[fmt][0](gs, n):
                want.add(-1)
            elif n % HEADER_RULES[fmt][1](gs):
                want.add(-2)
        if min(E, D, F, s, k) < 1 or max(D, F) > 51200 or s * k > 4096:
            want.add(-2)
        if not want and max(D, F) > 36864:
            want = {-2, -4}            # the shared-memory budget, checked with the launch shape
        want = want or {-4}
        got = L.qexpert_group_act(fmt, gs, None, None, None, None, None, None, E, D, F, None, s, k, None, None,
                                  act, limit, None, None, 0, None, None)
        assert got in want, (fmt, gs, E, D, F, s, k, act, limit, got, want)
        seen[got] += 1
    assert min(seen[-1], seen[-2], seen[-4], seen[-9]) >= 100, dict(seen)


def test_product_path_needs_no_oracle_and_has_no_fallback(L, tmp_path):
    """The package imports and loads its library with the oracle made
    unimportable; with the library missing, the first call raises instead of
    computing anything on the host."""
    import subprocess
    import sys
    pkg_dir = os.path.join(ROOT, "weight_only_quantized_qgemv_gb300")
    for fn in os.listdir(pkg_dir):
        if fn.endswith(".py"):
            text = open(os.path.join(pkg_dir, fn)).read()
            assert not re.search(r"^\s*(from|import)\s+oracle\b", text, flags=re.M), fn
    code = (
        "import sys\n"
        "sys.modules['oracle'] = None\n"
        "import weight_only_quantized_qgemv_gb300 as q\n"
        "from weight_only_quantized_qgemv_gb300 import _build, _lib\n"
        "assert _lib.lib() is not None\n"
        "_lib._lib = None\n"
        f"_build.LIB = {str(tmp_path / 'missing.so')!r}\n"
        "try:\n"
        "    q.qgemv(4, 32, 0, 0, 0, 16, 1024, 1, 0)\n"
        "except RuntimeError as e:\n"
        "    assert 'no CPU fallback' in str(e), e\n"
        "    print('raised')\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("raised")
