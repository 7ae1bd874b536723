"""The C-ABI library loads and exports every function include/*.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(det_[A-Za-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from deterministic_floating_point_gb300 import _build, det
    _build.build()
    return det.lib()


def test_header_declares_the_five_calls():
    names = declared_functions()
    for fn in ("det_sum", "det_scatter_add", "det_scatter_add_rows", "det_scan", "det_segmented_scan",
               "det_read_status", "det_status_string"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(declared_functions()) if getattr(lib, n, None) is None]
    assert not missing, missing


def test_status_strings(lib):
    from deterministic_floating_point_gb300 import det
    assert det.status_string(0) == "ok"
    for code in range(1, 8):
        assert det.status_string(code) != "unknown status"


def test_host_argument_checks_need_no_gpu(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)            # never dereferenced: the checks fail first
    assert lib.det_sum(fake, 10, 7, fake, fake, 1 << 20, 0, None) == 2          # dtype
    assert lib.det_sum(None, 10, 0, fake, fake, 1 << 20, 0, None) == 1          # null x
    assert lib.det_sum(fake, -1, 0, fake, fake, 1 << 20, 0, None) == 1          # n < 0
    assert lib.det_sum(fake, 10, 0, fake, fake, 1 << 20, 96, None) == 1         # block size
    assert lib.det_sum(fake, 10, 0, fake, vp((1 << 20) + 8), 1 << 20, 0, None) == 4  # misaligned ws


def test_workspace_queries_are_host_only(lib):
    assert lib.det_sum_workspace_bytes(0, 0) >= 256
    assert lib.det_sum_workspace_bytes(1 << 36, 0) > lib.det_sum_workspace_bytes(1 << 20, 0)
    assert lib.det_scan_workspace_bytes(1 << 28, 0) > lib.det_scan_workspace_bytes(1 << 20, 0)
    assert lib.det_scatter_add_workspace_bytes(1 << 24, 1024, 0) > 4 * (1 << 24)
    assert lib.det_sum_workspace_bytes(-1, 0) == 0


def test_host_checks_of_the_next_calls(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    # det_scan_i32: unknown flag bits, null input, misaligned workspace
    assert lib.det_scan_i32(fake, fake, 10, 2, None, fake, 1 << 20, 0, None) == 1
    assert lib.det_scan_i32(None, fake, 10, 0, None, fake, 1 << 20, 0, None) == 1
    assert lib.det_scan_i32(fake, fake, 10, 0, None, vp((1 << 20) + 8), 1 << 20, 0, None) == 4
    # det_slot_alloc: null counter with counters, negative n, too many records
    assert lib.det_slot_alloc(None, 4, fake, 0, None, 10, fake, fake, 1 << 20, 0, None) == 1
    assert lib.det_slot_alloc(fake, 4, fake, 0, None, -1, fake, fake, 1 << 20, 0, None) == 1
    assert lib.det_slot_alloc(fake, 4, fake, 0, None, 1 << 31, fake, fake, 1 << 40, 0, None) == 3
    # det_scatter_min / max: dtype, small workspace
    assert lib.det_scatter_min(fake, 4, fake, fake, 10, 9, fake, 1 << 20, 0, None) == 2
    assert lib.det_scatter_max(fake, 1 << 20, fake, fake, 10, 0, fake, 64, 0, None) == 4
    # det_scatter_sub shares det_scatter_add's checks
    assert lib.det_scatter_sub(fake, 4, None, fake, 10, 0, None, None, fake, 1 << 20, 0, None) == 1
    assert lib.det_scan_i32_workspace_bytes(1 << 20) > 0 and lib.det_slot_alloc_workspace_bytes(1 << 20, 4) > 0
    assert lib.det_scatter_minmax_workspace_bytes(1000, 1) >= 8000


def test_scan_withhold_hook_checks_its_limit(lib):
    assert lib.det_test_scan_withhold(5, 0) == 1                 # no limit
    assert lib.det_test_scan_withhold(5, 3 * 10**9) == 1         # above the 2 s default
    assert lib.det_test_scan_withhold(-1, 0) == 0                # clearing always works


def test_no_cpu_path_when_the_library_is_missing(tmp_path):
    """With libdet.so absent every call raises: nothing falls back to CPU code."""
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import torch\n"
        "from deterministic_floating_point_gb300 import det\n"
        "det.LIB_PATH = %r\n"
        "det._lib = None\n"
        "try:\n"
        "    det.lib()\n"
        "except RuntimeError as e:\n"
        "    print('raised', 'missing' in str(e))\n"
    ) % (ROOT, str(tmp_path / "absent" / "libdet.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "raised True"


def test_host_tensors_are_refused(lib):
    """The binding takes device tensors only; host tensors raise before any call."""
    import torch
    from deterministic_floating_point_gb300 import det
    x = torch.ones(16)
    for call in (lambda: det.det_sum(x), lambda: det.det_scan(x),
                 lambda: det.det_scatter_add(torch.zeros(4), torch.zeros(16, dtype=torch.int32), x)):
        with pytest.raises(ValueError):
            call()
