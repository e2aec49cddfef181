"""The C-ABI library on the CPU: it loads, exports every function include/fa.h declares, and
rejects bad arguments on the host before any CUDA work (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FA_OK, FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_DTYPE, FA_ERR_ALIGN, FA_ERR_ALIAS = 0, -1, -2, -3, -4, -5
FA_ERR_ARCH, FA_ERR_SCALE, FA_ERR_CUDA = -6, -9, -10


@pytest.fixture(scope="module")
def lib():
    from io_aware_attention_fa2_gb300 import build as fa_build
    from io_aware_attention_fa2_gb300 import binding
    fa_build.build()
    return binding.load_library()


def declared_functions():
    names = []
    for fname in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s+(fa_\w+)\s*\(", text, flags=re.M)
    return names


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"fa_fwd", "fa_error_string", "fa_get_device_error", "fa_abi_version"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    assert lib.fa_abi_version() == 1


def test_error_strings(lib):
    for code in range(-12, 1):
        assert lib.fa_error_string(code) != b"unknown status"
    assert lib.fa_error_string(-8) == b"a kernel wait ran past its limit"
    assert lib.fa_error_string(12345) == b"unknown status"


def _call(lib, q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, B=1, H=1, N=128,
          d=64, causal=0, scale=0.125, dtype=0):
    # Fake, never dereferenced addresses: every case below fails a host-side check first.
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, None)


def test_host_side_argument_checks(lib):
    assert _call(lib, q=0) == FA_ERR_NULL
    assert _call(lib, lse=0) == FA_ERR_NULL
    assert _call(lib, B=0) == FA_ERR_SHAPE
    assert _call(lib, N=0) == FA_ERR_SHAPE
    assert _call(lib, H=-1) == FA_ERR_SHAPE
    for d in (0, 32, 96, 256):
        assert _call(lib, d=d) == FA_ERR_SHAPE
    assert _call(lib, B=1 << 12, H=1 << 8, N=1 << 20) == FA_ERR_SHAPE   # >= 2^31 CTAs
    assert _call(lib, B=1 << 16, H=1 << 15) == FA_ERR_SHAPE   # B*H >= 2^31
    assert _call(lib, dtype=2) == FA_ERR_DTYPE
    assert _call(lib, scale=float("nan")) == FA_ERR_SCALE
    assert _call(lib, scale=float("inf")) == FA_ERR_SCALE
    assert _call(lib, q=0x10008) == FA_ERR_ALIGN
    assert _call(lib, o=0x40004) == FA_ERR_ALIGN
    assert _call(lib, lse=0x50002) == FA_ERR_ALIGN
    # o overlapping q (N=128, d=64 bf16: 16 KiB per tensor)
    assert _call(lib, o=0x10000 + 0x2000) == FA_ERR_ALIAS
    assert _call(lib, lse=0x30000 + 0x100) == FA_ERR_ALIAS
    assert _call(lib, lse=0x40000 + 0x100) == FA_ERR_ALIAS


def test_valid_arguments_without_gpu_fail_in_device_query(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover real launches")
    assert _call(lib) in (FA_ERR_CUDA, FA_ERR_ARCH)


def _split(lib, q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, B=1, H=1, Nq=16,
           Nk=128, d=64, causal=0, wl=-1, wr=-1, lens=None, scale=0.125, dtype=0, splits=2,
           ws=0x100000, ws_bytes=1 << 20):
    # Fake, never dereferenced addresses: every case below fails a host-side check first.
    return lib.fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, causal, wl, wr, lens, scale,
                              dtype, splits, ws, ws_bytes, None)


def test_splitkv_workspace_size_and_split_count(lib):
    # [num_splits, B, H, Nq, d] fp32 parts + [num_splits, B, H, Nq] fp32 LSE
    assert lib.fa_fwd_splitkv_workspace_size(2, 3, 5, 128, 4) == 4 * 2 * 3 * 5 * (128 + 1) * 4
    assert lib.fa_fwd_splitkv_workspace_size(2, 3, 5, 128, 1) == 0
    # enough (b, h, Q block) units for every SM: no split
    assert lib.fa_fwd_splitkv_num_splits(2, 16, 8192, 8192, 152) == 1
    # decoding, 64K keys (512 tiles): waves x (tiles per part + 4) is smallest at 7 parts for
    # 128 heads (6 waves x 78) and at 9 parts for 32 heads (2 waves x 61)
    assert lib.fa_fwd_splitkv_num_splits(4, 32, 1, 65536, 152) == 7
    assert lib.fa_fwd_splitkv_num_splits(4, 8, 1, 65536, 152) == 9
    # few keys: parts keep at least 2 tiles
    assert lib.fa_fwd_splitkv_num_splits(1, 1, 1, 1024, 152) == 4
    assert lib.fa_fwd_splitkv_num_splits(1, 1, 1, 100, 152) == 1
    assert lib.fa_fwd_splitkv_num_splits(1, 1, 1, 1 << 30, 152) == 128


def test_splitkv_host_side_checks(lib):
    assert _split(lib, Nk=8) == FA_ERR_SHAPE                 # Nk < Nq
    assert _split(lib, splits=0) == FA_ERR_SHAPE
    assert _split(lib, splits=129) == FA_ERR_SHAPE
    assert _split(lib, ws=0) == FA_ERR_NULL                  # parts need a workspace
    assert _split(lib, ws_bytes=100) == -11                  # FA_ERR_WORKSPACE
    assert _split(lib, ws=0x100008) == FA_ERR_ALIGN
    assert _split(lib, ws=0x40000) == FA_ERR_ALIAS           # workspace over o
    assert _split(lib, ws=0x20000) == FA_ERR_ALIAS           # workspace over k
    assert lib.fa_error_string(-11) == b"workspace smaller than fa_fwd_splitkv_workspace_size()"


def _noalloc(lib, q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000, B=1, H=1, Nq=16,
             Nk=128, d=64, causal=0, wl=-1, wr=-1, lens=None, scale=0.125, dtype=0, splits=2):
    # Fake, never dereferenced addresses: every case below fails a host-side check first.
    fn = lib.fa_fwd_splitkv_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, f32, i32, i32,
                   vp]
    fn.restype = i32
    return fn(q, k, v, o, lse, B, H, Nq, Nk, d, causal, wl, wr, lens, scale, dtype, splits, None)


def test_noalloc_checks_arguments_like_splitkv(lib):
    """fa_fwd_splitkv_noalloc gives fa_fwd_splitkv's codes for bad arguments, before it looks
    at its built-in buffer: a split count beyond the limit is a shape error even when its
    parts would not fit the buffer either."""
    assert _noalloc(lib, q=0) == FA_ERR_NULL
    assert _noalloc(lib, splits=129) == FA_ERR_SHAPE
    assert _noalloc(lib, splits=129, B=64, H=64, Nq=256) == FA_ERR_SHAPE
    assert _noalloc(lib, splits=0) == FA_ERR_SHAPE
    assert _noalloc(lib, Nk=8) == FA_ERR_SHAPE
    assert _noalloc(lib, dtype=5) == FA_ERR_DTYPE
    assert _noalloc(lib, scale=float("nan")) == FA_ERR_SCALE
    assert _noalloc(lib, q=0x10008) == FA_ERR_ALIGN
    assert _noalloc(lib, o=0x10000) == FA_ERR_ALIAS


def test_fwd_host_host_side_checks(lib):
    # Fake, never dereferenced addresses: every case below fails a host-side check first.
    h = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000]
    dvc = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000]

    def call(hosts=h, devs=dvc, B=2, H=1, N=128, d=64, dtype=0):
        return lib.fa_fwd_host(*hosts, *devs, B, H, N, d, 0, 0.125, dtype, None)

    assert call(hosts=[0] + h[1:]) == FA_ERR_NULL
    assert call(hosts=h[:4] + [0]) == FA_ERR_NULL
    assert call(devs=[0] + dvc[1:]) == FA_ERR_NULL
    assert call(B=0) == FA_ERR_SHAPE
    assert call(d=96) == FA_ERR_SHAPE
    assert call(dtype=5) == FA_ERR_DTYPE
    assert call(devs=[0x10008] + dvc[1:]) == FA_ERR_ALIGN
    assert call(devs=dvc[:3] + [0x10000 + 0x100, dvc[4]]) == FA_ERR_ALIAS   # o_d over q_d


def test_selftest_wait_timeout_host_checks(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == FA_ERR_SHAPE
    assert lib.fa_selftest_wait_timeout(2000001, None) == FA_ERR_SHAPE
    import torch
    if not torch.cuda.is_available():
        assert lib.fa_selftest_wait_timeout(1000, None) in (FA_ERR_CUDA, FA_ERR_ARCH)


def test_fwd_host_device_buffers_disjoint(lib):
    # the host entry point writes q_d, k_d, v_d itself, so inputs may not share memory either
    h = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000]
    dvc = [0x10000, 0x10000 + 0x100, 0x30000, 0x40000, 0x50000]       # k_d over q_d
    assert lib.fa_fwd_host(*h, *dvc, 2, 1, 128, 64, 0, 0.125, 0, None) == FA_ERR_ALIAS


def test_bwd_host_host_side_checks(lib):
    # Fake, never dereferenced addresses: every case below fails a host-side check first.
    # B=2, H=1, N=128, d=64: 32 KiB per tensor, 65 KiB of workspace; buffers 1 MiB apart.
    h = [0x1000 * (i + 1) for i in range(9)]
    dvc = [0x100000 * (i + 1) for i in range(9)]
    ws, ws_bytes = 0x100000 * 10, int(lib.fa_bwd_workspace_size(2, 1, 128, 64))

    def call(hosts=h, devs=dvc, w=ws, wb=ws_bytes, B=2, N=128, d=64, dtype=0):
        return lib.fa_bwd_host(*hosts, *devs, w, wb, B, 1, N, d, 0, 0.125, dtype, None)

    assert call(hosts=h[:8] + [0]) == FA_ERR_NULL
    assert call(hosts=[0] + h[1:]) == FA_ERR_NULL
    assert call(devs=dvc[:4] + [0] + dvc[5:]) == FA_ERR_NULL
    assert call(w=0) == FA_ERR_NULL
    assert call(B=0) == FA_ERR_SHAPE
    assert call(d=256) == FA_ERR_SHAPE
    assert call(dtype=7) == FA_ERR_DTYPE
    assert call(wb=ws_bytes - 4) == -11                                  # FA_ERR_WORKSPACE
    assert call(devs=dvc[:6] + [dvc[6] + 8] + dvc[7:]) == FA_ERR_ALIGN   # dq_d
    assert call(devs=dvc[:4] + [dvc[3] + 0x100] + dvc[5:]) == FA_ERR_ALIAS   # do_d over o_d
    assert call(devs=dvc[:1] + [dvc[0] + 0x100] + dvc[2:]) == FA_ERR_ALIAS   # k_d over q_d
    assert call(w=dvc[8] + 0x100) == FA_ERR_ALIAS                        # workspace over dv_d


def test_bwd_masked_host_side_checks(lib):
    # Fake, never dereferenced addresses; B=2, H=1, N=128, d=64: 32 KiB per tensor.
    ptrs = [0x100000 * (i + 1) for i in range(9)]
    ws, ws_bytes = 0x100000 * 10, int(lib.fa_bwd_workspace_size(2, 1, 128, 64))

    def call(lens=0, left=-1, right=-1):
        return lib.fa_bwd_masked(*ptrs, 2, 1, 128, 64, 1, left, right, lens, 0.125, 0, ws,
                                 ws_bytes, None)

    assert call(lens=0x2000002) == FA_ERR_ALIGN                 # key lengths not 4-byte aligned
    assert call(lens=ptrs[6] + 64) == FA_ERR_ALIAS              # key lengths inside dq
    # the unmasked call reaches the same checks as the masked one with no mask
    assert lib.fa_bwd(*ptrs, 2, 1, 0, 64, 0, 0.125, 0, ws, ws_bytes, None) == FA_ERR_SHAPE


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/fa.h compiles as strict C99 (no CUDA headers needed: the stream is an opaque
    pointer) and a C program calling through it links against the built library."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from io_aware_attention_fa2_gb300 import build as fa_build
    src = tmp_path / "use_fa.c"
    src.write_text('#include "fa.h"\n#include <stdio.h>\n'
                   'int main(void) {\n'
                   '  printf("%d %s\\n", fa_abi_version(), fa_error_string(FA_ERR_SHAPE));\n'
                   '  return fa_abi_version() == 1 ? 0 : 1;\n}\n')
    exe = tmp_path / "use_fa"
    lib_path = fa_build.build()
    libdir = os.path.dirname(lib_path)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", libdir, "-l:" + os.path.basename(lib_path),
           "-Wl,-rpath," + libdir]
    subprocess.run(cmd, check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    assert out.split()[0] == "1" and "unsupported shape" in out


def test_host_masked_entry_points_host_checks(lib):
    # Fake, never dereferenced addresses: every case below fails a host-side check first.
    h = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000]
    dvc = [0x100000, 0x200000, 0x300000, 0x400000, 0x500000]

    def fwd(lens=0, hosts=h):
        return lib.fa_fwd_host_masked(*hosts, *dvc, 2, 1, 128, 64, 1, 32, 0, lens, 0.125, 0,
                                      None)

    assert fwd(hosts=[0] + h[1:]) == FA_ERR_NULL
    assert fwd(lens=0x600002) == FA_ERR_ALIGN                   # key lengths not 4-byte aligned
    assert fwd(lens=dvc[3] + 64) == FA_ERR_ALIAS                # key lengths inside o_d
    hb = [0x1000 * (i + 1) for i in range(9)]
    db = [0x100000 * (i + 1) for i in range(9)]
    ws, ws_bytes = 0x100000 * 10, int(lib.fa_bwd_workspace_size(2, 1, 128, 64))

    def bwd(lens=0):
        return lib.fa_bwd_host_masked(*hb, *db, ws, ws_bytes, 2, 1, 128, 64, 0, 16, 16, lens,
                                      0.125, 0, None)

    assert bwd(lens=0xB00002) == FA_ERR_ALIGN
    assert bwd(lens=db[7] + 64) == FA_ERR_ALIAS                 # key lengths inside dk_d
