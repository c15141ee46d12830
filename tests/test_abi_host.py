"""Host-side contract of the C ABI (no GPU needed).

Checks that libsn builds for sm_103a, loads, exports every function that
include/sn_abi.h declares, and honours the version / capability / status
rules of "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时" §6
(packed version, sn_abi_check refuses a foreign major, unknown capability
bits ignored, int32 status codes).  Calls with a NULL context must fail with
SN_E_INVAL before touching the device.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sn_abi.h")


@pytest.fixture(scope="module")
def abi():
    from scan_runtime_gb300 import _build, _abi
    _build.build()
    _abi.load()
    return _abi


def _header_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sn_[a-z0-9_]+)\s*\(", src)))


def _header_defines():
    out = {}
    for m in re.finditer(r"#define\s+(SN_[A-Z0-9_]+)\s+\(?\s*(-?\d+)(u)?\s*(<<\s*(\d+))?\)?", open(HEADER).read()):
        v = int(m.group(2))
        if m.group(5):
            v <<= int(m.group(5))
        out[m.group(1)] = v
    return out


def test_header_declares_the_five_compute_calls():
    fns = _header_functions()
    for f in ("sn_scan_fma", "sn_scan_gated", "sn_recur_diag", "sn_recur_delta", "sn_recur_rwkv7",
              "sn_abi_check", "sn_abi_caps", "sn_abi_version"):
        assert f in fns


def test_library_exports_every_declared_symbol(abi):
    lib = abi.load()
    fns = _header_functions()
    for f in fns:
        assert hasattr(lib, f), f"{f} declared in sn_abi.h but not exported"
    assert set(fns) == set(abi.EXPORTS)
    nm = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (sn_\w+)", nm))
    assert set(fns) <= exported


def test_binding_constants_match_header(abi):
    d = _header_defines()
    for name, val in d.items():
        if name.startswith(("SN_ABI_VERSION", "SN_OK", "SN_E_", "SN_CAP_", "SN_DECAY_", "SN_OPT_",
                            "SN_SCAN_KERNEL_", "SN_OP_")) and hasattr(abi, name):
            assert getattr(abi, name) == val, name


def test_version_packing_and_check(abi):
    assert abi.sn_abi_version() == (1 << 16) | (0 << 8) | 0
    assert abi.sn_abi_check(abi.SN_ABI_VERSION_MAJOR) == abi.SN_OK
    for bad in (0, 2, -1, 1 << 16):
        assert abi.sn_abi_check(bad) == abi.SN_E_UNSUPPORTED


def test_caps_bits(abi):
    caps = abi.sn_abi_caps()
    for bit in (abi.SN_CAP_SCAN_FMA, abi.SN_CAP_SCAN_GATED, abi.SN_CAP_RECUR_DIAG, abi.SN_CAP_RECUR_DELTA,
                abi.SN_CAP_RECUR_RWKV7, abi.SN_CAP_DECODE, abi.SN_CAP_SCAN_LOOKBACK, abi.SN_CAP_SCAN_BACKWARD,
                abi.SN_CAP_RECUR_CHUNKED, abi.SN_CAP_READOUT, abi.SN_CAP_DELTA_CHUNKED):
        assert caps & bit
    assert caps & ~0x7FF == 0           # no undocumented bits set


def test_status_strings(abi):
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert abi.sn_status_str(s) and abi.sn_status_str(s) != "unknown status"
    assert abi.sn_status_str(-99) == "unknown status"


def test_null_context_is_rejected_before_any_device_work(abi):
    E = abi.SN_E_INVAL
    x = 0x1000                           # never dereferenced: the NULL context fails first
    assert abi.sn_scan_fma(None, 1, 1, 4, x, x, None, None, x, 0) == E
    assert abi.sn_scan_gated(None, 1, 1, 4, x, x, None, None, x, 0) == E
    assert abi.sn_recur_diag(None, 1, 1, 1, 1, 64, 64, 0, 1.0, x, x, x, x, None, None, x, 0) == E
    assert abi.sn_recur_delta(None, 1, 1, 1, 64, 64, 1.0, x, x, x, x, None, None, x, 0) == E
    assert abi.sn_recur_rwkv7(None, 1, 1, 1, 64, 64, x, x, x, x, None, None, x, 0) == E
    assert abi.sn_scan_fma_backward(None, 1, 1, 4, x, None, x, x, None, x, x, x, 0) == E
    assert abi.sn_scan_gated_backward(None, 1, 1, 4, x, x, None, x, x, None, x, x, x, 0) == E
    assert abi.sn_ctx_set_option(None, abi.SN_OPT_SCAN_KERNEL, 0) == E
    assert abi.sn_ctx_get_option(None, abi.SN_OPT_SCAN_KERNEL)[0] == E
    assert abi.sn_ctx_last_error(None) == E
    assert abi.sn_ctx_set_workspace(None, None, 0) == E
    abi.sn_ctx_free(None)               # no-op


def test_ctx_create_argument_errors(abi):
    lib = abi.load()
    assert lib.sn_ctx_create(0, None) == abi.SN_E_INVAL
    s, h = abi.sn_ctx_create(-1)
    assert s != abi.SN_OK and not h.value


def test_ctx_create_without_gpu_fails_cleanly(abi):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    s, h = abi.sn_ctx_create(0)
    assert s in (abi.SN_E_DEVICE, abi.SN_E_INVAL) and not h.value


def test_workspace_bytes(abi):
    nb = abi.sn_workspace_bytes(abi.SN_OP_SCAN_FMA, 8, 8192, 2048)
    tiles = 8 * (2048 // 32) * (8192 // 128)
    # flags, the A and B aggregates (f32) and the tagged carry words (u64)
    lb = ((tiles * 4 + 255) // 256) * 256 + tiles * (2 * 32 * 4 + 32 * 8)
    # the fused kernel's tagged words (from eight chunks on), chunks padded to
    # groups of four: 256 bytes of group-end carries and 2048 of aggregates
    # per group and column, then the initial carries
    cols, chunks = 8 * (2048 // 32), 8192 // 128
    assert nb == max(lb, cols * (2304 * ((chunks + 3) // 4) + 256))
    cols, chunks = 3 * (64 // 32), 9
    fused = cols * (2304 * ((chunks + 3) // 4) + 256)
    lb = ((cols * chunks * 4 + 255) // 256) * 256 + cols * chunks * 512
    assert fused > lb
    assert abi.sn_workspace_bytes(abi.SN_OP_SCAN_FMA, 3, 9 * 128, 64) == fused
    # fewer than ten chunks: the reduce-then-scan arrays (chunks in groups of
    # four per column, three arrays, plus the columns' initial carries) set it
    cols, chunks = 2 * (64 // 32), 5
    flags = ((cols * chunks * 4 + 255) // 256) * 256
    rs = 3 * cols * ((chunks + 3) // 4) * 32 * 4 * 4 + cols * 32 * 4
    assert rs > cols * chunks * 512
    assert abi.sn_workspace_bytes(abi.SN_OP_SCAN_FMA, 2, 5 * 128, 64) == flags + rs
    assert abi.sn_workspace_bytes(abi.SN_OP_SCAN_GATED, 1, 1, 1) > 0
    assert abi.sn_workspace_bytes(99, 1, 1, 1) == -1
    assert abi.sn_workspace_bytes(abi.SN_OP_SCAN_FMA, 0, 1, 1) == -1
    assert abi.sn_workspace_bytes(abi.SN_OP_SCAN_FMA, 1, -5, 1) == -1
    # dimensions whose product exceeds the element bound (or int64): -1, no overflow
    big = 2 ** 31 - 1
    assert abi.sn_workspace_bytes(abi.SN_OP_SCAN_FMA, big, big, big) == -1
    assert abi.sn_recur_chunked_workspace_bytes(big, big, big, 128, 128) == -1
    assert abi.sn_recur_delta_chunked_workspace_bytes(big, big, 1, 128, 128) == -1


def test_scan_host_staging_bytes(abi):
    r256 = lambda x: (x + 255) // 256 * 256
    for B, T, N, mask, rows in ((8, 8192, 2048, 3, 1), (5, 300, 192, 1, 2), (3, 7, 5, 2, 9)):
        forms = (mask & 1) + ((mask >> 1) & 1)
        r = min(rows, B)
        slot = r256(r * T * N * 4) + r256(r * N * 4) + forms * (2 * r256(r * T * N * 4) + r256(r * N * 4))
        assert abi.sn_scan_host_staging_bytes(B, T, N, mask, rows) == 3 * slot
    assert abi.sn_scan_host_staging_bytes(1, 1, 1, 0, 1) == -1
    assert abi.sn_scan_host_staging_bytes(1, 1, 1, 4, 1) == -1
    assert abi.sn_scan_host_staging_bytes(1, 1, 1, 1, 0) == -1
    assert abi.sn_scan_host_staging_bytes(2 ** 31 - 1, 2 ** 31 - 1, 2 ** 31 - 1, 1, 1) == -1


def test_chunked_workspace_bytes(abi):
    r256 = lambda x: (x + 255) // 256 * 256
    for B, T, H, dv in ((4, 4096, 4, 128), (1, 300, 3, 64), (2, 1, 1, 128)):
        nc = (T + 127) // 128
        # chunk states, the chunk decays and anchor factors, one flag per chunk,
        # and the chunk's v tile (transposed once, for the output stage)
        want = (r256(B * H * nc * 128 * dv * 4) + 2 * r256(B * H * nc * 128 * 4) + r256(B * H * nc * 4) +
                r256(B * H * nc * dv * 128 * 4))
        assert abi.sn_recur_chunked_workspace_bytes(B, T, H, 128, dv) == want


def test_noalloc_rejects_oversized_problems_before_any_device_work(abi):
    """Dimensions whose element count overflows int64 are an argument error,
    found before the device is touched (the pointers are never read)."""
    big = 2 ** 31 - 1
    fake = 1 << 20
    for B, T, N in ((big, big, big), (4, big, big), (1, 1 << 20, 1 << 21)):
        assert abi.sn_scan_lookback_noalloc(0, B, T, N, fake, fake, None, None, None, None, 0) == abi.SN_E_INVAL


def test_product_package_does_not_touch_the_oracle():
    """The CUDA path never imports the oracle: scan the product sources."""
    pkg = os.path.join(ROOT, "scan_runtime_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"\boracle\b", src), f"{f} mentions the oracle"
