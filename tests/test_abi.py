"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, and rejects bad arguments on the host before touching CUDA."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_77_gb300 import build, ops

    build.build()
    return ops.load_library()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("spec_select_topk", "spec_verify_attn", "spec_verify_attn_sparse", "spec_lse_merge",
                 "spec_select_workspace_size", "spec_verify_workspace_size", "spec_read_device_status"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_verification_77_gb300 import ops

    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in ops.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert lib.spec_status_string(0) == b"SPEC_OK"
    assert lib.spec_status_string(5) == b"SPEC_ERR_BAD_INPUT"
    assert lib.spec_status_string(99) == b"SPEC_ERR_UNKNOWN"
    assert lib.spec_last_cuda_error() == b"no error"  # nothing has failed in this thread


def test_workspace_sizes(lib):
    a = lib.spec_verify_workspace_size(4, 64, 32, 8, 128, 32768)
    b = lib.spec_verify_workspace_size(8, 64, 32, 8, 128, 32768)
    assert 256 < a < b
    assert lib.spec_verify_workspace_size(1, 1, 3, 2, 128, 10) == 0  # Hq % Hkv != 0
    assert lib.spec_select_workspace_size(16, 32768, 2048) >= 4


def _verify_args(**over):
    F = ctypes.c_float
    args = dict(q=16, kc=16, vc=16, sb=0, sh=0, st=128, kd=None, vd=None, par=None, B=1, N=1, Hq=1, Hkv=1,
                d=128, L=4, ctx=None, scale=F(0.1), out=16, lse=16, ws=256, ws_bytes=1 << 30, stream=None)
    args.update(over)
    return list(args.values())


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1),                      # null pointer
    (dict(N=0), 1),                         # no draft node
    (dict(Hq=3, Hkv=2), 1),                 # Hq % Hkv != 0
    (dict(q=24), 1),                        # misaligned
    (dict(kd=16, vd=None), 1),              # draft K without V
    (dict(kd=16, vd=16, par=None), 1),      # draft block without parents
    (dict(st=100), 1),                      # stride not a multiple of 8
    (dict(ws=128), 1),                      # workspace not 256-aligned
    (dict(d=64), 2),                        # head_dim other than 128
])
def test_verify_rejects_bad_arguments_on_the_host(lib, over, code):
    # fake, never-dereferenced addresses: the checks return before any CUDA call
    assert lib.spec_verify_attn(*_verify_args(**over)) == code


@pytest.mark.parametrize("over,code", [
    (dict(budget=0), 1), (dict(sink=3, window=3, budget=5), 1), (dict(L=0), 1),
    (dict(ld=10, L=20), 1), (dict(top_m=-1), 1), (dict(idx=None), 1), (dict(L=2_000_000, ld=2_000_000), 1),
])
def test_select_rejects_bad_arguments_on_the_host(lib, over, code):
    a = dict(ds=16, ts=16, ld=100, B=1, L=100, ctx=None, sink=1, window=1, top_m=2, budget=10, idx=16,
             count=None, ws=256, ws_bytes=256, stream=None)
    a.update(over)
    assert lib.spec_select_topk(*a.values()) == code


@pytest.mark.parametrize("over,code", [
    (dict(tok=None), 1), (dict(N=0), 1), (dict(N=5000), 1), (dict(tok=18), 1),  # null, N out of range, misaligned
    (dict(kc=16), 1),                              # commit arguments given only in part
    (dict(kc=16, vc=16, kd=16, vd=16, ctx=16, d=64), 2),   # head_dim other than 128
    (dict(kc=16, vc=16, kd=16, vd=16, ctx=16, st=100), 1),  # stride not a multiple of 8
    (dict(kc=24, vc=16, kd=16, vd=16, ctx=16), 1),          # cache not 16-byte aligned
])
def test_accept_rejects_bad_arguments_on_the_host(lib, over, code):
    a = dict(tok=16, par=16, tn=16, B=1, N=4, path=16, ln=16, bonus=16, kc=None, vc=None, sb=0, sh=0, st=128,
             kd=None, vd=None, Hkv=1, d=128, L=8, ctx=None, status=None, stream=None)
    a.update(over)
    assert lib.spec_accept_commit(*a.values()) == code


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(B=0), 1), (dict(B=70000), 1), (dict(Hq=3), 1), (dict(ld=10), 1),
    (dict(st=100), 1), (dict(q=24), 1), (dict(d=64), 2), (dict(N=600), 2),
])
def test_importance_rejects_bad_arguments_on_the_host(lib, over, code):
    a = dict(q=16, kc=16, sb=0, sh=0, st=128, lse=16, heads=16, nh=1, B=1, N=4, Hq=4, Hkv=2, d=128, L=64,
             ctx=None, scale=ctypes.c_float(0.1), score=16, ld=64, status=None, stream=None)
    a.update(over)
    assert lib.spec_importance_scores(*a.values()) == code


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(N=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(st=100), 1), (dict(q=24), 1),
    (dict(d=64), 2),
    # 64 sequences x 1 KV head x (2^31 - 1) / 64 + 1 tiles = 2^31 tiles: beyond 32-bit tile numbering
    (dict(B=64, L=2**31 - 1), 2),
])
def test_noalloc_rejects_bad_arguments_on_the_host(lib, over, code):
    # fake, never-dereferenced addresses: every one of these checks returns before any CUDA call
    a = dict(q=16, kc=16, vc=16, sb=0, sh=0, st=128, kd=None, vd=None, par=None, B=1, N=1, Hq=1, Hkv=1, d=128,
             L=4, ctx=None, scale=ctypes.c_float(0.1), out=16, lse=16, status=None, stream=None)
    a.update(over)
    assert lib.spec_verify_attn_noalloc(*a.values()) == code


@pytest.mark.parametrize("over,code", [
    (dict(bs=0), 1), (dict(ld=1, L=300), 1), (dict(st=0), 1), (dict(d=64), 2), (dict(sb=1001), 1),
    (dict(dtype=7), 1),
    # sparse: the block stride must be a multiple of the row stride (pool rows are numbered)
    (dict(idx=16, budget=4, sb=1032, st=16), 2),
])
def test_paged_rejects_bad_arguments_on_the_host(lib, over, code):
    # fake, never-dereferenced addresses: every one of these checks returns before any CUDA call
    from speculative_decoding_verification_77_gb300 import ops

    e = dict(table=16, ld=4, bs=128, nblk=8, dtype=0)
    for k in e:
        if k in over:
            e[k] = over.pop(k)
    ext = ops._VerifyExt(e["table"], e["ld"], e["bs"], e["nblk"], e["dtype"])
    a = dict(q=16, kp=16, vp=16, sb=128 * 128, sh=128 * 128, st=128, kd=None, vd=None, par=None, B=1, N=1, Hq=1,
             Hkv=1, d=128, L=300, ctx=None, scale=ctypes.c_float(0.1), idx=None, budget=0, ext=ctypes.byref(ext),
             out=16, lse=16, ws=256, ws_bytes=1 << 30, stream=None)
    a.update(over)
    assert lib.spec_verify_attn_ex(*a.values()) == code


@pytest.mark.parametrize("over,code", [
    (dict(kvd=7), 1), (dict(ks=None), 1), (dict(vs=None), 1), (dict(ks=18), 1),
    # fp8 rows are copied 16 bytes at a time: strides (bytes) must be multiples of 16
    (dict(st=136), 1), (dict(sh=1000), 1),
])
def test_fp8_rejects_bad_arguments_on_the_host(lib, over, code):
    # fake, never-dereferenced addresses: every one of these checks returns before any CUDA call
    from speculative_decoding_verification_77_gb300 import ops

    e = dict(kvd=1, ks=16, vs=16)
    for k in e:
        if k in over:
            e[k] = over.pop(k)
    ext = ops._VerifyExt(None, 0, 0, 0, 0, e["kvd"], e["ks"], e["vs"])
    a = dict(q=16, kc=16, vc=16, sb=300 * 128, sh=300 * 128, st=128, kd=None, vd=None, par=None, B=1, N=1, Hq=1,
             Hkv=1, d=128, L=300, ctx=None, scale=ctypes.c_float(0.1), idx=None, budget=0, ext=ctypes.byref(ext),
             out=16, lse=16, ws=256, ws_bytes=1 << 30, stream=None)
    a.update(over)
    assert lib.spec_verify_attn_ex(*a.values()) == code


def test_merge_rejects_bad_arguments_on_the_host(lib):
    assert lib.spec_lse_merge(None, 4, 4, 4, 4, 4, 10, 128, None) == 1
    assert lib.spec_lse_merge(4, 4, 4, 4, 4, 4, -1, 128, None) == 1
    assert lib.spec_lse_merge(4, 4, 4, 4, 4, 4, 10, 0, None) == 1
    assert lib.spec_lse_merge(4, 4, 4, 4, 4, 4, 8 * (2**31 - 1) + 1, 128, None) == 1  # past the grid's reach


def test_package_import_loads_nothing():
    import importlib
    import sys

    mod = importlib.import_module("speculative_decoding_verification_77_gb300")
    assert "speculative_decoding_verification_77_gb300.ops" not in sys.modules or mod is not None


def test_product_does_not_use_the_oracle():
    """The product package must neither import nor call the oracle."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_77_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    src = f.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), fn
                assert "spec_oracle" not in src and "oracle_attend" not in src, fn


def test_binding_refuses_cpu_tensors(lib):
    """No CPU fallback anywhere: every tensor entry point of the binding rejects host tensors."""
    import torch

    from speculative_decoding_verification_77_gb300 import ops

    bf = lambda *s: torch.zeros(s, dtype=torch.bfloat16)
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)
    f32 = lambda *s: torch.zeros(s, dtype=torch.float32)
    calls = [
        lambda: ops.select_topk(f32(1, 64), f32(1, 64), sink=1, window=1, top_m=2, budget=8),
        lambda: ops.verify_attn(bf(1, 2, 4, 128), bf(1, 2, 16, 128), bf(1, 2, 16, 128)),
        lambda: ops.verify_attn_sparse(bf(1, 2, 4, 128), bf(1, 2, 16, 128), bf(1, 2, 16, 128), None, None, None,
                                       i32(1, 8)),
        lambda: ops.lse_merge(f32(2, 128), f32(2), f32(2, 128), f32(2)),
        lambda: ops.accept_commit(i32(1, 4), i32(1, 4), i32(1, 5)),
        lambda: ops.importance_scores(bf(1, 2, 4, 128), bf(1, 2, 16, 128), f32(1, 2, 4), i32(1)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def test_header_is_plain_c_and_links(lib, tmp_path):
    """The header compiles as strict C99 (a C caller needs no C++ or torch), and a C program links
    the library and calls a host-only entry point (no GPU needed)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text('#include "specverify.h"\n'
                   "int main(void) {\n"
                   "    int32_t starts[600], info[8];\n"
                   "    int ctas = spec_split_plan(4, 64, 32, 8, 32768, 152, 0, starts, 600, info);\n"
                   "    return (ctas == 152 && starts[0] == 0 && starts[ctas] == info[0] * info[1]) ? 0 : 1;\n"
                   "}\n")
    libdir = os.path.join(ROOT, "speculative_decoding_verification_77_gb300")
    exe = tmp_path / "caller"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lspecverify", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert subprocess.run([str(exe)], timeout=60).returncode == 0
