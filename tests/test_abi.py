"""The C-ABI library builds for sm_103a, loads, exports every declared symbol,
and rejects bad arguments on the host (no GPU needed, no compute calls)."""
import ctypes

import pytest

import balanced_tree_build_gb300 as kdt
from balanced_tree_build_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kdt.lib()


def test_exports_every_header_symbol(lib):
    names = kdt.header_symbols()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_workspace_size_argument_checks(lib):
    out = ctypes.c_size_t(0)
    for n, k, mode in [(0, 3, 0), (-5, 3, 0), (2**31, 3, 0), (10, 0, 0), (10, kdt_max_k() + 1, 0),
                       (10, 3, 2), (10, 3, -1)]:
        assert lib.kdt_workspace_size(n, k, mode, ctypes.byref(out)) == kdt.EINVAL, (n, k, mode)
    assert lib.kdt_workspace_size(10, 3, 0, None) == kdt.EINVAL
    assert lib.kdt_workspace_size(2**31 - 1, 3, 0, ctypes.byref(out)) == kdt.OK


def kdt_max_k():
    with open(kdt.HEADER_PATH) as f:
        for line in f:
            if line.startswith("#define KDT_MAX_K"):
                return int(line.split()[2])
    raise AssertionError("KDT_MAX_K not found")


def test_workspace_grows_with_n(lib):
    sizes = [kdt.workspace_bytes(n, 3, 0) for n in (1, 1000, 10**6, 10**8)]
    assert sizes == sorted(sizes)
    # two record buffers of k keys + 1 index per point dominate
    assert sizes[-1] >= 2 * 4 * 4 * 10**8
    assert kdt.host_workspace_bytes(1000, 3, 0) > kdt.workspace_bytes(1000, 3, 0)


def test_build_rejects_bad_arguments_before_touching_the_device(lib):
    fake = ctypes.c_void_p(0x1000)
    assert lib.kdt_build(None, 10, 3, 0, fake, None) == kdt.EINVAL
    assert lib.kdt_build(fake, 10, 3, 0, None, None) == kdt.EINVAL
    assert lib.kdt_build(fake, 0, 3, 0, fake, None) == kdt.EINVAL
    assert lib.kdt_build(fake, 10, 3, 7, fake, None) == kdt.EINVAL
    assert lib.kdt_build_ws(fake, 10, 3, 0, fake, None, 1 << 20, None) == kdt.EINVAL
    need = kdt.workspace_bytes(10, 3, 0)
    assert lib.kdt_build_ws(fake, 10, 3, 0, fake, ctypes.c_void_p(0x100000), need - 1, None) == kdt.ENOMEM
    assert lib.kdt_build_ws(fake, 10, 3, 0, fake, ctypes.c_void_p(0x100001), need, None) == kdt.EINVAL
    assert lib.kdt_verify(None, 10, 3, 0, fake, None) == kdt.EINVAL
    assert lib.kdt_verify(fake, 10, 3, 5, fake, None) == kdt.EINVAL
    assert lib.kdt_build_host(None, 10, 3, 0, fake, fake, 1 << 30, None) == kdt.EINVAL


def test_error_strings(lib):
    for code in (kdt.OK, kdt.EINVAL, kdt.ENOMEM, kdt.ECUDA, kdt.ENONFINITE, kdt.ETIMEOUT, kdt.EINTERNAL):
        s = lib.kdt_error_string(code)
        assert s and s != b"unknown error"
    assert lib.kdt_error_string(12345) == b"unknown error"


def test_profile_switch_without_launches(lib):
    kdt.profile_enable(True)
    kdt.profile_reset()
    assert kdt.profile_read() == []
    kdt.profile_enable(False)


def test_kernel_stat_struct_matches_the_header(lib):
    """The ctypes mirror of kdt_kernel_stat has the header's fields, in order,
    with the same widths (the binding reads the array the library fills)."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(kdt.__file__), os.pardir, "include", "kdtree_build.h")).read()
    body = re.search(r"typedef struct \{([^}]*)\} kdt_kernel_stat;", hdr).group(1)
    fields = re.findall(r"^\s*([A-Za-z_][A-Za-z_0-9 ]*?)\s*\*?\s*([A-Za-z_][A-Za-z_0-9]*);", body, re.M)
    ctype_of = {"const char": ctypes.c_char_p, "int64_t": ctypes.c_int64, "double": ctypes.c_double}
    want = [(name, ctype_of[t.strip()]) for t, name in fields]
    assert kdt._KernelStat._fields_ == want
    assert ctypes.sizeof(kdt._KernelStat) == 40


def test_balanced_entry_points_argument_checks(lib):
    out = ctypes.c_int64(0)
    for n, want in [(1, 1), (2, 3), (3, 3), (4, 7), (1000, 1023), (2**31 - 1, 2**31 - 1)]:
        assert lib.kdt_balanced_slots(n, ctypes.byref(out)) == kdt.OK
        assert out.value == want
    assert lib.kdt_balanced_slots(0, ctypes.byref(out)) == kdt.EINVAL
    assert lib.kdt_balanced_slots(10, None) == kdt.EINVAL
    sz = ctypes.c_size_t(0)
    assert lib.kdt_balanced_workspace_size(10, 3, ctypes.byref(sz)) == kdt.OK and sz.value > 0
    assert lib.kdt_balanced_workspace_size(10, kdt_max_k() + 1, ctypes.byref(sz)) == kdt.EINVAL
    fake = ctypes.c_void_p(0x1000)
    assert lib.kdt_build_balanced(None, 10, 3, fake, fake, 1 << 20, None) == kdt.EINVAL
    assert lib.kdt_build_balanced(fake, 10, 3, fake, ctypes.c_void_p(0x100000), 1, None) == kdt.ENOMEM
