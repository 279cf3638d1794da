"""C-ABI checks that need no GPU: the library builds, loads, exports every symbol that
include/attn.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from exact_attention_forward_attn_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    assert _declared_functions() == sorted(
        ["attn_fwd", "attn_status_string", "attn_last_cuda_error", "attn_debug_status",
         "attn_fwd_num_splits", "attn_fwd_test_split_choice",
         "attn_fwd_splitkv", "attn_fwd_splitkv_workspace_bytes", "attn_fwd_splitkv_num_splits",
         "attn_fwd_splitkv_noalloc", "attn_fwd_splitkv_noalloc_max_bytes", "attn_fwd_strided",
         "attn_fwd_test_stall", "attn_fwd_test_kernel", "attn_bwd", "attn_bwd_workspace_bytes",
         "attn_mla_decode",
         "attn_mla_decode_test_stall", "attn_mla_decode_num_splits",
         "attn_mla_decode_workspace_bytes"])


def test_library_exports_every_declared_symbol(lib):
    nm = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", nm, re.M))
    for name in _declared_functions():
        assert name in exported, f"{name} declared in attn.h but not exported"
        assert callable(getattr(lib, name))
    assert set(_lib.SIGNATURES) == set(_declared_functions())


def test_debug_build_exports_every_declared_symbol():
    """The index-checking debug build (ATTN_DEBUG) compiles and exports the same boundary."""
    path = build.build(debug=True)
    nm = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                        check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", nm, re.M))
    assert set(_declared_functions()) <= exported


def test_built_for_sm_103a_only():
    cmd = build.nvcc_command("/dev/null")
    assert "arch=compute_103a,code=sm_103a" in cmd
    assert sum(1 for c in cmd if c == "-gencode") == 1


def test_status_strings(lib):
    for st in range(-15, 1):
        s = lib.attn_status_string(st)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.attn_status_string(0) == b"ok"
    assert lib.attn_status_string(12345) == b"unknown status"


# Host-side validation returns before any CUDA call; fake, aligned, never-dereferenced addresses.
P = 0x10000


def _call(lib, q=P, k=P * 2, v=P * 3, out=P * 4, lse=P * 5, B=1, Hq=2, Hkv=1, N=128, D=64,
          causal=0, scale=0.125):
    return lib.attn_fwd(q, k, v, out, lse, B, Hq, Hkv, N, D, causal, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), -1), (dict(out=0), -1), (dict(lse=0), -1),
    (dict(B=-1), -2), (dict(N=-5), -2), (dict(Hq=0), -2), (dict(Hkv=0), -2),
    (dict(Hq=6, Hkv=4), -3),
    (dict(D=100), -4), (dict(D=264), -4), (dict(D=0), -4), (dict(D=512), -4), (dict(D=4), -4),
    (dict(D=252), -4),
    (dict(scale=0.0), -6), (dict(scale=-1.0), -6), (dict(scale=float("inf")), -6),
    (dict(scale=float("nan")), -6),
    (dict(q=P + 8), -5), (dict(lse=P * 5 + 4), -5),
])
def test_host_validation(lib, kw, status):
    assert _call(lib, **kw) == status


def test_empty_problem_is_a_no_op(lib):
    assert _call(lib, B=0) == 0
    assert _call(lib, N=0) == 0
    # zero-size tensors often have NULL data pointers
    assert _call(lib, B=0, q=0, k=0, v=0, out=0, lse=0) == 0
    assert _call(lib, N=0, q=0, k=0, v=0, out=0, lse=0) == 0
    # shape errors still win over the empty shortcut
    assert _call(lib, B=0, Hq=3, Hkv=2) == -3


def test_aliasing_output_is_rejected(lib):
    # out overlapping q: rejected before any device query
    assert _call(lib, out=P) == -11
    assert _call(lib, lse=P * 4 + 64) == -11


S = 1 << 24  # fake addresses 16 MiB apart (larger than any tensor below)


def _split(lib, q=S, k=S * 2, v=S * 3, out=S * 4, lse=S * 5, B=1, Hq=2, Hkv=1, N=512, D=64,
           causal=0, scale=0.125, splits=2, ws=S * 8, ws_bytes=1 << 30):
    return lib.attn_fwd_splitkv(q, k, v, out, lse, B, Hq, Hkv, N, D, causal,
                                ctypes.c_float(scale), splits, ws, ws_bytes, None)


def test_splitkv_workspace_bytes(lib):
    # n_splits * B*Hq * N * (D + 1) * 4 bytes, with the split count the tile layout allows
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 32, 512, 128, 2) == 2 * 32 * 512 * 129 * 4
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 16, 512, 128, 4) == 4 * 16 * 512 * 129 * 4
    # 4 key tiles into 3 requested splits -> 2 tiles per split -> 2 splits
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 32, 512, 128, 3) == 2 * 32 * 512 * 129 * 4
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 32, 512, 128, 1) == 0
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 2, 100, 64, 8) == 0  # one key tile
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 2, 128, 100, 2) == 0  # bad D
    # padded head dims: partials are 64 or 128 wide
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 32, 512, 96, 2) == 2 * 32 * 512 * 129 * 4
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 32, 512, 32, 2) == 2 * 32 * 512 * 65 * 4


@pytest.mark.parametrize("kw,status", [
    (dict(splits=-1), -12), (dict(splits=65), -12),
    (dict(ws=0), -1), (dict(ws=S * 8 + 4), -5), (dict(ws_bytes=1000), -13),
    (dict(ws=S), -11),  # workspace overlaps q
    (dict(Hq=3, Hkv=2), -3), (dict(D=36), -4),
])
def test_splitkv_host_validation(lib, kw, status):
    assert _split(lib, **kw) == status


def test_splitkv_empty_problem(lib):
    assert _split(lib, B=0, ws=0, ws_bytes=0) == 0


def _strided(lib, qs=(2 * 128 * 64, 128 * 64, 64), ks=(128 * 64, 128 * 64, 64),
             os_=(2 * 128 * 64, 128 * 64, 64), B=1, Hq=2, Hkv=1, N=128, D=64):
    arr = lambda t: (ctypes.c_longlong * 3)(*t) if t is not None else None
    return lib.attn_fwd_strided(S, S * 2, S * 3, S * 4, S * 5, B, Hq, Hkv, N, D, 0,
                                ctypes.c_float(0.125), arr(qs), arr(ks), arr(ks), arr(os_), None)


@pytest.mark.parametrize("kw,status", [
    (dict(qs=None), -1), (dict(ks=(0, 8192, 64)), -15), (dict(os_=(16384, 8192, 68)), -15),
    (dict(qs=(16384, -8192, 64)), -15), (dict(qs=(16384, 8192, 12)), -15),
])
def test_strided_host_validation(lib, kw, status):
    assert _strided(lib, **kw) == status


def test_bwd_workspace_bytes(lib):
    assert lib.attn_bwd_workspace_bytes(2, 8, 1000) == 2 * 8 * 1000 * 4
    assert lib.attn_bwd_workspace_bytes(0, 8, 1000) == 0


def _mla(lib, q=S, kv=S * 2, out=S * 4, lse=S * 5, B=1, H=128, T=4096, d_c=512, d_r=64,
         scale=192 ** -0.5, splits=8, ws=S * 8, ws_bytes=1 << 30):
    # 8 splits: above the cluster merge's 4, so the workspace is needed and checked
    return lib.attn_mla_decode(q, kv, out, lse, B, H, T, d_c, d_r, ctypes.c_float(scale), splits,
                               ws, ws_bytes, None)


def test_mla_workspace_bytes(lib):
    # above 4 splits n_splits * B * H * (512 + 1) fp32 (each split's O and LSE); 2-4 splits merge
    # inside a cluster and need none; splits are clamped to the 64-token tiles
    assert lib.attn_mla_decode_workspace_bytes(2, 128, 4096, 8) == 8 * 2 * 128 * 513 * 4
    assert lib.attn_mla_decode_workspace_bytes(2, 128, 4096, 5) == 5 * 2 * 128 * 513 * 4
    assert lib.attn_mla_decode_workspace_bytes(2, 128, 4096, 4) == 0
    assert lib.attn_mla_decode_workspace_bytes(1, 16, 100, 8) == 0  # clamped to 2 splits
    assert lib.attn_mla_decode_workspace_bytes(1, 16, 64, 8) == 0  # one tile: no split
    assert lib.attn_mla_decode_workspace_bytes(1, 16, 4096, 1) == 0
    assert lib.attn_mla_decode_workspace_bytes(0, 16, 4096, 4) == 0
    assert lib.attn_mla_decode_workspace_bytes(1, 16, 4096, 65) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), -1), (dict(lse=0), -1), (dict(ws=0), -1),
    (dict(B=-1), -2), (dict(H=0), -2), (dict(T=0), -2),
    (dict(d_c=256), -4), (dict(d_r=32), -4),
    (dict(q=S + 8), -5), (dict(ws=S * 8 + 4), -5),
    (dict(scale=0.0), -6), (dict(scale=float("nan")), -6),
    (dict(out=S + 64), -11), (dict(ws=S * 2), -11),
    (dict(splits=-1), -12), (dict(splits=65), -12),
    (dict(ws_bytes=1000), -13),
])
def test_mla_host_validation(lib, kw, status):
    assert _mla(lib, **kw) == status


def test_mla_empty_batch_is_a_no_op(lib):
    assert _mla(lib, B=0, q=0, kv=0, out=0, lse=0, ws=0, ws_bytes=0) == 0


def test_wide_heads_are_forward_only(lib):
    # the backward holds at most 128 columns: D = 192 is rejected before anything else
    assert lib.attn_bwd(S, S * 2, S * 3, S * 4, S * 5, S * 6, S * 7, S * 8, S * 9, 1, 2, 1, 128, 192,
                        0, ctypes.c_float(0.1), S * 10, 1 << 20, None) == -4
    # the test hook lives in the two-tile kernel only
    assert lib.attn_fwd_test_stall(S, S * 2, S * 3, S * 4, S * 5, 1, 2, 1, 128, 256, 0,
                                   ctypes.c_float(0.1), 0, None) == -4
    # split-KV with wide heads runs as one split: no workspace
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 32, 4096, 256, 4) == 0


def test_kernel_hook_rejects_what_its_kernels_do_not_run(lib):
    def call(D, kernel):
        return lib.attn_fwd_test_kernel(S, S * 2, S * 3, S * 4, S * 5, 1, 2, 1, 128, D, 0,
                                        ctypes.c_float(0.1), kernel, -1, None)
    assert call(128, 0) == -2 and call(128, 4) == -2   # no such kernel: ATTN_ERR_SHAPE
    assert call(256, 1) == -4 and call(256, 2) == -4   # wide heads: none of them
    assert call(256, 3) == -4
    assert call(64, 2) == -4                           # the pair kernel is for D in (64, 128]
