"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before any CUDA call. Nothing here launches a kernel or
touches a device (all pointers are fake and every case fails validation)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mamba_ssm.h")


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_125_b300 import build, binding
    build.build()
    return binding.library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MAMBA_API\s+[\w\s\*]*?\b(mamba_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    for required in ("mamba_selective_scan_fwd", "mamba_selective_state_update"):
        assert required in names
    from selective_state_space_125_b300 import binding
    assert sorted(binding.EXPORTED) == names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} not exported"


def test_only_the_abi_is_exported():
    from selective_state_space_125_b300 import binding
    out = os.popen(f"nm -D --defined-only {binding.LIB_PATH}").read().split("\n")
    names = {line.split()[-1] for line in out if line.strip() and " T " in line}
    assert {n for n in names if n.startswith("mamba_")} == set(declared_symbols())


def test_version_and_strings(lib):
    assert lib.mamba_version() >= 10000
    for code, word in [(0, b"ok"), (1, b"invalid"), (2, b"unsupported"), (3, b"CUDA"), (4, b"timed out")]:
        assert word in lib.mamba_status_string(code)


FAKE = 0x7F0000000000  # never dereferenced: every call below fails validation


def scan(lib, batch=2, dim=8, dstate=16, seqlen=4, dtype=1, u=FAKE, delta=FAKE + 0x100000,
         A_log=FAKE + 0x200000, B=FAKE + 0x300000, C=FAKE + 0x400000, D=None, z=None, bias=None,
         h0=None, out=FAKE + 0x500000, last=None, plan=None):
    return lib.mamba_selective_scan_fwd_ex(batch, dim, dstate, seqlen, dtype, u, delta, A_log, B, C, D,
                                           z, bias, h0, out, last, plan, None)


@pytest.mark.parametrize("kw,status", [
    (dict(batch=-1), 1), (dict(dim=-3), 1), (dict(seqlen=-1), 1), (dict(dstate=0), 1),
    (dict(dstate=257), 2), (dict(dtype=7), 1), (dict(batch=70000), 2),
    (dict(u=None), 1), (dict(delta=None), 1), (dict(B=None), 1), (dict(C=None), 1),
    (dict(out=None), 1), (dict(A_log=None), 1),
    (dict(out=FAKE), 1),                                   # out aliases u
    (dict(last=FAKE + 0x300000 + 8), 1),                   # last_state aliases B
])
def test_scan_rejects_bad_arguments(lib, kw, status):
    assert scan(lib, **kw) == status
    assert lib.mamba_last_error_detail() != b""


def test_bad_plan_knobs(lib):
    from selective_state_space_125_b300.binding import ScanPlan
    for p in (ScanPlan(-1, 0, 0), ScanPlan(0, -2, 0), ScanPlan(0, 0, 3), ScanPlan(0, 0, 0, 2),
              ScanPlan(0, 0, 0, -1)):
        assert scan(lib, plan=ctypes.byref(p)) == 1


def test_state_update_rejects_unknown_discretisation(lib):
    assert lib.mamba_selective_state_update_ex(2, 8, 16, 1, FAKE, FAKE + 0x100000, FAKE + 0x200000,
                                               FAKE + 0x300000, FAKE + 0x400000, FAKE + 0x500000, None, None,
                                               None, FAKE + 0x600000, 5, None) == 1


def test_empty_problems_are_ok_without_a_device(lib):
    # batch == 0 or dim == 0: nothing to do, no CUDA call is made.
    assert scan(lib, batch=0) == 0
    assert scan(lib, dim=0) == 0
    assert lib.mamba_selective_state_update(0, 8, 16, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                            None, None, None, FAKE + 0x900000, None) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(batch=-1), 1), (dict(dstate=0), 1), (dict(dstate=300), 2), (dict(dtype=5), 1),
    (dict(state=None), 1), (dict(u=None), 1), (dict(out=None), 1),
    (dict(out=FAKE), 1),                                   # out aliases state
])
def test_state_update_rejects_bad_arguments(lib, kw, status):
    a = dict(batch=2, dim=8, dstate=16, dtype=1, state=FAKE, u=FAKE + 0x100000, delta=FAKE + 0x200000,
             A_log=FAKE + 0x300000, B=FAKE + 0x400000, C=FAKE + 0x500000, out=FAKE + 0x600000)
    a.update(kw)
    assert lib.mamba_selective_state_update(a["batch"], a["dim"], a["dstate"], a["dtype"], a["state"], a["u"],
                                            a["delta"], a["A_log"], a["B"], a["C"], None, None, None,
                                            a["out"], None) == status


def test_binding_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    from selective_state_space_125_b300 import binding
    x = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        binding.mamba_selective_scan_fwd(x, x, torch.zeros(8, 16), torch.zeros(1, 4, 16), torch.zeros(1, 4, 16))
    with pytest.raises(TypeError):
        binding.mamba_selective_scan_fwd(x.double(), x, torch.zeros(8, 16), x, x)


def test_conv_scan_rejects_bad_arguments(lib):
    from selective_state_space_125_b300.binding import ScanPlan
    args = lambda width, w=FAKE + 0x700000, plan=None: (2, 8, 16, 4, 1, FAKE, w, None, width, FAKE + 0x100000,
                                                        FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, None,
                                                        None, None, None, FAKE + 0x500000, None, plan, None)
    assert lib.mamba_conv1d_selective_scan_fwd(*args(5)) == 2          # width > 4
    assert lib.mamba_conv1d_selective_scan_fwd(*args(0)) == 2          # width < 1
    assert lib.mamba_conv1d_selective_scan_fwd(*args(4, w=None)) == 1  # no taps
    p = ScanPlan(0, 0, 0, 1)
    assert lib.mamba_conv1d_selective_scan_fwd(*args(4, plan=ctypes.byref(p))) == 2  # simplified + conv


def _bwd_args(batch=2, dim=8, dstate=16, seqlen=4, dtype=1, disc=0, **over):
    """Arguments of mamba_selective_scan_bwd with distinct fake 16-byte-aligned pointers."""
    names = ["u", "delta", "A_log", "B", "C", "D", "z", "delta_bias", "initial_state", "dout", "dlast_state",
             "du", "ddelta", "dA_log", "dB", "dC", "dD", "dz", "ddelta_bias", "dinitial_state"]
    ptrs = {n: FAKE + (i + 1) * 0x1000000 for i, n in enumerate(names)}
    for opt in ("D", "z", "delta_bias", "initial_state", "dlast_state", "dD", "dz", "ddelta_bias",
                "dinitial_state"):
        ptrs[opt] = None
    ptrs.update(over)
    return (batch, dim, dstate, seqlen, dtype, disc) + tuple(ptrs[n] for n in names) + (None,)


@pytest.mark.parametrize("kw,status", [
    (dict(dstate=8), 2),                          # not built for this state size
    (dict(dstate=256), 2),
    (dict(disc=2), 1),                            # unknown discretisation
    (dict(dtype=7), 1),
    (dict(seqlen=-1), 1),
    (dict(dstate=0), 1),
    (dict(batch=70000), 2),
    (dict(dz=FAKE + 0x30000000), 1),              # dz without z
    (dict(du=None), 1),                           # required output missing
    (dict(dout=None), 1),
    (dict(dA_log=FAKE + 0xE000004), 2),          # fp32 gradient array not 16-byte aligned
    (dict(initial_state=FAKE + 0x9000008), 2),
    (dict(du=FAKE + 0x1000000), 1),               # du is u
    (dict(dB=FAKE + 0xC000010), 1),               # dB overlaps du
])
def test_bwd_rejects_bad_arguments(lib, kw, status):
    over = {k: v for k, v in kw.items() if k not in ("batch", "dim", "dstate", "seqlen", "dtype", "disc")}
    sizes = {k: v for k, v in kw.items() if k in ("batch", "dim", "dstate", "seqlen", "dtype", "disc")}
    assert lib.mamba_selective_scan_bwd(*_bwd_args(**sizes, **over)) == status


def test_bwd_empty_problem_is_ok_without_a_device(lib):
    # nothing to zero and nothing to launch
    assert lib.mamba_selective_scan_bwd(*_bwd_args(batch=0, dim=0)) == 0


def test_bwd_ex_rejects_negative_segments(lib):
    args = _bwd_args()
    assert lib.mamba_selective_scan_bwd_ex(*args[:-1], -1, None) == 1


C_CLIENT = r"""
#include <stdio.h>
#include "mamba_ssm.h"
int main(void) {
    int v = mamba_version();
    /* every call below is rejected by validation, before any CUDA call */
    mamba_status_t s1 = mamba_selective_scan_bwd(1, 8, 8, 4, MAMBA_BF16, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0,
                                                 0, 0, 0, 0, 0, 0, 0, 0, 0);
    mamba_status_t s2 = mamba_selective_scan_fwd(-1, 8, 16, 4, MAMBA_BF16, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);
    mamba_status_t s3 = mamba_selective_state_update_ex(1, 8, 16, MAMBA_F32, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 7, 0);
    printf("%d %d %d %d %s\n", v, (int)s1, (int)s2, (int)s3, mamba_last_error_detail());
    return 0;
}
"""


def test_plain_c_client_links_and_calls_the_abi(lib, tmp_path):
    """The library is a C ABI: a C99 program (no Python, no torch) compiles against the
    header, links the shared library and gets its statuses."""
    import subprocess
    from selective_state_space_125_b300 import binding
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(binding.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lmamba_ssm_b300", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == lib.mamba_version()
    assert out[1:4] == ["2", "1", "1"]  # unsupported N; negative size; unknown discretisation
