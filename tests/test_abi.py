"""The C-ABI library without a GPU: it loads, exports what include/dq4.h declares,
and validates arguments on the host before touching CUDA."""

import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dq4.h")


@pytest.fixture(scope="module")
def dq():
    from quantized_weight_dequantization_gb300 import build
    build.build()
    import quantized_weight_dequantization_gb300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(dq4\w*)\s*\(", text, flags=re.M)))


def _declared_constants():
    text = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(DQ4_\w+)\s+(\d+)", text)}


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == sorted(["dq4_abi_version", "dq4_nested", "dq4_nested_transposed", "dq4",
                            "dq4_nested_unfused",
                            "dq4_nested_unfused_static", "dq4_status_string",
                            "dq4_int8_correction_prep", "dq4_nested_out_prod",
                            "dq4_nested_linear", "dq4_nested_linear_workspace_bytes",
                            "dq4_nested_out_prod_workspace_bytes",
                            "dq4_nested_host", "dq4_nested_host_scratch_bytes",
                            "dq4_last_cuda_error"]), names


def test_library_exports_every_declared_symbol(dq):
    from quantized_weight_dequantization_gb300.build import LIB_PATH
    lib = ctypes.CDLL(LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                        text=True)
    if nm.returncode == 0:
        exported = {line.split()[-1] for line in nm.stdout.splitlines() if " T " in line}
        for name in _declared_functions():
            assert name in exported, name


def test_header_constants_match_binding(dq):
    c = _declared_constants()
    from quantized_weight_dequantization_gb300._binding import STATUS_NAMES
    for code, name in STATUS_NAMES.items():
        assert c[name] == code
    assert (c["DQ4_OUT_F16"], c["DQ4_OUT_BF16"], c["DQ4_OUT_F32"]) == (dq.OUT_F16, dq.OUT_BF16,
                                                                       dq.OUT_F32)


def test_status_strings(dq):
    for code in range(0, 12):
        s = dq.lib.dq4_status_string(code)
        assert s and s != b"unknown status", code
    assert dq.lib.dq4_status_string(1234) == b"unknown status"
    assert dq.lib.dq4_abi_version() == 3


def test_host_validation_before_any_cuda_call(dq):
    L = dq.lib
    nz = 1 << 12  # any nonzero fake pointer: never dereferenced on these paths
    args = dict(packed=nz, codes=nz, absmax=nz, scb=nz, vcb=nz, off=0.0, n=100, bs=64, nbs=256,
                dt=0, out=nz, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return L.dq4_nested(a["packed"], a["codes"], a["absmax"], a["scb"], a["vcb"], a["off"],
                            a["n"], a["bs"], a["nbs"], a["dt"], a["out"], a["stream"])

    assert call(n=-1) == 2
    for bs in (0, 16, 48, 8192, -64):
        assert call(bs=bs) == 3, bs
    for nbs in (0, 3, -256):
        assert call(nbs=nbs) == 4, nbs
    for dt in (-1, 3, 7):
        assert call(dt=dt) == 5, dt
    assert call(n=0, packed=None, codes=None, absmax=None, scb=None, vcb=None, out=None) == 0
    for k in ("packed", "codes", "absmax", "scb", "vcb", "out"):
        assert call(**{k: None}) == 1, k
    assert call(absmax=nz + 2) == 6
    assert call(out=nz + 1) == 6
    assert call(dt=2, out=nz + 2) == 6
    # non-nested and unfused forms
    assert L.dq4(nz, nz, nz, 10, 33, 0, nz, None) == 3
    assert L.dq4(nz, None, nz, 10, 64, 0, nz, None) == 1
    assert L.dq4(nz, nz, nz, 0, 64, 0, nz, None) == 0
    assert L.dq4_nested_unfused(nz, nz, nz, nz, nz, 0.0, 10, 64, 256, 0, nz, None, None) == 1
    assert L.dq4_nested_unfused(nz, nz, nz, nz, nz, 0.0, 10, 64, 256, 0, nz, nz + 1, None) == 6
    # transposed form: rows / cols validated on the host
    T = L.dq4_nested_transposed
    assert T(nz, nz, nz, nz, nz, 0.0, -1, 8, 64, 256, 0, nz, None) == 2
    assert T(nz, nz, nz, nz, nz, 0.0, 8, -1, 64, 256, 0, nz, None) == 2
    assert T(nz, nz, nz, nz, nz, 0.0, 1 << 40, 1 << 40, 64, 256, 0, nz, None) == 2
    assert T(None, None, None, None, None, 0.0, 0, 77, 64, 256, 0, None, None) == 0
    assert T(nz, nz, nz, nz, nz, 0.0, 8, 8, 48, 256, 0, nz, None) == 3
    assert T(nz, None, nz, nz, nz, 0.0, 8, 8, 64, 256, 0, nz, None) == 1
    assert T(nz, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, 0, nz + 1, None) == 6
    # LLM.int8 preparation: shapes and pointers validated on the host
    P = L.dq4_int8_correction_prep
    assert P(nz, nz, nz, nz, -1, 4, 4, 2, nz, nz, None, None) == 2
    assert P(nz, nz, nz, nz, 4, 4, 0, 2, nz, nz, None, None) == 2
    assert P(None, None, None, None, 4, 4, 4, 0, None, None, None, None) == 0
    assert P(nz, nz, nz, None, 4, 4, 4, 2, nz, nz, None, None) == 1
    assert P(None, nz, nz, nz, 4, 4, 4, 2, nz, nz, None, None) == 1
    assert P(nz, nz, nz, nz + 4, 4, 4, 4, 2, nz, nz, None, None) == 6
    assert P(nz, nz, nz + 2, nz, 4, 4, 4, 2, nz, nz, None, None) == 6
    # row-blocked dequant fused into a GEMM: shape, workspace and pointers on the host
    O = L.dq4_nested_out_prod
    assert O(nz, nz, nz, nz, nz, 0.0, -1, 8, 64, 256, nz, 4, nz, nz, 1 << 20, None, None) == 2
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, nz, 0, nz, nz, 1 << 20, None, None) == 0
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 256, 64, 256, nz, 4, nz, nz, -1, None, None) == 2
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, None, 4, nz, nz, 1 << 20, None, None) == 1
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, nz, 4, None, nz, 1 << 20, None, None) == 1
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 8, 48, 256, nz, 4, nz, nz, 1 << 20, None, None) == 3
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, nz, 4, nz, nz + 2, 1 << 20, None,
             None) == 6  # a workspace that is not 4-byte aligned
    assert O(nz, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, nz, 4, nz, nz, 1 << 20, nz + 2,
             None) == 6  # the failure counter likewise
    assert O(nz + 1, nz, nz, nz, nz, 0.0, 8, 8, 64, 256, nz, 4, nz, nz, 1 << 20, None,
             None) == 6  # packed is staged in 4-byte words
    assert L.dq4_nested_out_prod_workspace_bytes(0, 8, 8) == 0
    # fused dequant + GEMM: shapes, dtypes and alignment on the host
    Lr = L.dq4_nested_linear
    assert Lr(nz, 1, nz, nz, nz, nz, nz, 0.0, 4, 8, 100, 64, 256, 1, nz, None, 0, None, None) == 2
    assert Lr(nz, 2, nz, nz, nz, nz, nz, 0.0, 4, 8, 64, 64, 256, 1, nz, None, 0, None, None) == 5
    assert Lr(nz, 1, nz, nz, nz, nz, nz, 0.0, 0, 8, 64, 64, 256, 1, nz, None, 0, None, None) == 0
    assert Lr(None, 1, nz, nz, nz, nz, nz, 0.0, 4, 8, 64, 64, 256, 1, nz, None, 0, None,
              None) == 1
    assert Lr(nz + 8, 1, nz, nz, nz, nz, nz, 0.0, 4, 8, 64, 64, 256, 1, nz, None, 0, None,
              None) == 6
    assert Lr(nz, 1, nz, nz, nz, nz, nz, 0.0, 4, 8, 64, 64, 256, 1, nz, nz + 16, 1 << 20, None,
              None) == 6  # a workspace that is not 256-byte aligned
    assert L.dq4_nested_linear_workspace_bytes(4, 8, 100) == 0  # K not a multiple of 64
    # host-to-host form: arguments and the scratch size on the host
    H = L.dq4_nested_host
    need = L.dq4_nested_host_scratch_bytes(1 << 20, 64, 256, 0)
    assert need > 0 and L.dq4_nested_host_scratch_bytes(0, 64, 256, 0) == 0
    assert L.dq4_nested_host_scratch_bytes(100, 48, 256, 0) == 0  # bad blocksize
    assert H(nz, nz, nz, nz, nz, 0.0, -1, 64, 256, 0, nz, nz, need, None) == 2
    assert H(nz, nz, nz, nz, nz, 0.0, 0, 64, 256, 0, nz, nz, need, None) == 0
    assert H(nz, nz, nz, nz, nz, 0.0, 100, 64, 256, 0, nz, None, need, None) == 1
    assert H(nz, nz, nz, nz, nz, 0.0, 100, 64, 256, 0, nz, nz + 16, need, None) == 6
    assert H(nz, nz, nz, nz, nz, 0.0, 1 << 20, 64, 256, 0, nz, nz, 4096, None) == 10
    # allocation-free form: the static scratch limit is checked before anything else runs
    limit = _declared_constants()["DQ4_STATIC_SCRATCH_BLOCKS"]
    assert L.dq4_nested_unfused_static(nz, nz, nz, nz, nz, 0.0, 64 * limit + 1, 64, 256, 0, nz,
                                       None) == 10
    assert L.dq4_nested_unfused_static(nz, nz, nz, nz, nz, 0.0, 0, 64, 256, 0, nz, None) == 0
    assert L.dq4_nested_unfused_static(None, nz, nz, nz, nz, 0.0, 100, 64, 256, 0, nz, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device status")
def test_no_device_reports_device_error(dq):
    nz = 1 << 12
    st = dq.lib.dq4_nested(nz, nz, nz, nz, nz, 0.0, 10, 64, 256, 0, nz, None)
    assert st == 7  # DQ4_ERR_DEVICE: nothing was launched
    assert dq.lib.dq4_last_cuda_error() != 0


def test_binding_rejects_host_tensors(dq):
    t8 = torch.zeros(64, dtype=torch.uint8)
    f = torch.zeros(256, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dq.dq4_nested(t8, t8, f, f, f[:16], 0.0, 64, 64, 256)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dq.dq4(t8, f, f[:16], 64, 64)


def test_product_does_not_reference_the_oracle():
    """The package's sources never import or load anything from oracle/."""
    pkg = os.path.join(ROOT, "quantized_weight_dequantization_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                for pat in (r"\bimport\s+oracle\b", r"\bfrom\s+oracle\b", r"oracle/",
                            r"liboracle", r"oracle_\w+\s*\("):
                    assert not re.search(pat, text), (os.path.join(dirpath, fn), pat)
