"""The C-ABI library builds, loads without a GPU and exports what include/pa.h declares.

Only host-side paths run here: symbol lookup, workspace planning and argument
checks that return before any CUDA call.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_140_gb300 import _build, _lib
    _build.build()
    return _lib.load()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_copy_blocks", "pa_decode_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from paged_kv_cache_140_gb300 import _lib
    names = declared_functions()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_only_api_symbols_are_exported(lib):
    from paged_kv_cache_140_gb300 import _lib
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", _lib.lib_path()], capture_output=True, text=True).stdout
    funcs = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(declared_functions()) <= funcs
    extra = {f for f in funcs if not f.startswith("pa_") and not f.startswith("_")}
    assert not extra, f"unexpected exports: {sorted(extra)[:10]}"


def test_status_strings(lib):
    for s in range(6):
        assert lib.pa_status_string(s)
    assert lib.pa_version() >= 100


def test_workspace_planning(lib):
    # Single partition: no workspace.
    assert lib.pa_decode_workspace_size(4, 4, 4, 64, 16, 100, 0) == 0
    assert lib.pa_decode_partition_size(4, 4, 4, 64, 16, 100, 0) == 112
    # 13B-shaped: 256 seqs x 40 heads, 2048 tokens in 256-token partitions.
    P = lib.pa_decode_partition_size(256, 40, 40, 128, 16, 2048, 0)
    assert P == 256
    n = lib.pa_decode_workspace_size(256, 40, 40, 128, 16, 2048, 0)
    slots = 256 * 40 * 8
    assert n >= slots * 128 * 4 + slots * 2 * 4
    # GQA long context with the 512-token partitions.
    assert lib.pa_decode_partition_size(16, 32, 8, 128, 16, 32768, 512) == 512
    n = lib.pa_decode_workspace_size(16, 32, 8, 128, 16, 32768, 512)
    assert n >= 16 * 8 * 64 * 4 * (128 + 2) * 4
    # Rejected requests.
    bad = ctypes.c_size_t(-1).value
    assert lib.pa_decode_workspace_size(4, 6, 4, 64, 16, 100, 0) == bad     # Hq % Hkv != 0
    assert lib.pa_decode_workspace_size(4, 4, 4, 96, 16, 100, 0) == bad     # head_dim 96
    assert lib.pa_decode_workspace_size(4, 4, 4, 64, 12, 100, 0) == bad     # block_size 12
    assert lib.pa_decode_workspace_size(4, 4, 4, 64, 16, 100, 24) == bad    # partition not /16
    assert lib.pa_decode_workspace_size(4, 4, 4, 64, 8, 1000, 512) == bad   # > 32 blocks/partition


def test_argument_checks_return_before_touching_a_gpu(lib):
    from paged_kv_cache_140_gb300 import _lib as L
    nul = ctypes.c_void_p(0)
    # pa_decode: negative sizes, bad dtype, bad grouping, context bound beyond the table.
    def dec(out_dt, q_dt, kv_dt, maxnb, maxctx, B, hq, hkv, d, scale=0.1, ks=1.0, vs=1.0, bs=16):
        return lib.pa_decode(nul, out_dt, nul, q_dt, nul, nul, kv_dt, ks, vs, nul, maxnb, nul, maxctx, B, hq,
                             hkv, d, bs, 64, scale, 0, nul, 0, nul, nul)
    # pa_decode: negative sizes, bad dtype, bad grouping, context bound beyond the table.
    assert dec(2, 1, 1, 8, 100, -1, 4, 4, 64) == L.PA_ERR_INVALID_ARG
    assert dec(2, 2, 2, 8, 100, 4, 4, 4, 64) == L.PA_ERR_INVALID_ARG          # f32 query / cache
    assert dec(2, 1, 1, 8, 100, 4, 12, 4, 64) == L.PA_ERR_UNSUPPORTED         # group of 3
    assert dec(2, 1, 1, 4, 100, 4, 4, 4, 64) == L.PA_ERR_INVALID_ARG          # 100 > 4 * 16
    assert dec(2, 1, 1, 8, 100, 4, 4, 4, 64, scale=float("nan")) == L.PA_ERR_INVALID_ARG
    assert dec(2, 0, 1, 8, 100, 4, 4, 4, 64) == L.PA_ERR_UNSUPPORTED          # f16 query, bf16 cache
    assert dec(2, 1, 3, 8, 100, 4, 4, 4, 64) == L.PA_ERR_UNSUPPORTED          # fp8 cache needs D 128
    assert dec(2, 1, 3, 8, 100, 4, 4, 4, 128, ks=0.0) == L.PA_ERR_INVALID_ARG  # fp8 scale must be > 0
    # Null tensors with real work.
    assert dec(2, 1, 1, 8, 100, 4, 4, 4, 64) == L.PA_ERR_INVALID_ARG
    assert dec(2, 1, 3, 8, 100, 4, 4, 4, 128, ks=0.5, vs=0.5) == L.PA_ERR_INVALID_ARG
    # Empty batch is a no-op.
    assert dec(2, 1, 1, 8, 100, 0, 4, 4, 64) == L.PA_OK
    # reshape_and_cache / copy_blocks.
    def rc(T, dt, cdt, ks=1.0, vs=1.0):
        return lib.pa_reshape_and_cache(nul, nul, nul, nul, nul, T, 64, 16, 4, 64, dt, cdt, ks, vs, nul, nul)
    assert rc(0, 0, 0) == L.PA_OK
    assert rc(3, 0, 0) == L.PA_ERR_INVALID_ARG                # null tensors
    assert rc(3, 2, 2) == L.PA_ERR_INVALID_ARG                # f32 rows
    assert rc(3, 0, 1) == L.PA_ERR_UNSUPPORTED                # f16 rows into a bf16 cache
    assert rc(3, 1, 3, ks=-1.0) == L.PA_ERR_INVALID_ARG       # fp8 scale must be > 0
    assert rc(3, 1, 3, ks=0.25, vs=0.25) == L.PA_ERR_INVALID_ARG  # null tensors
    assert lib.pa_copy_blocks(nul, nul, nul, 0, 64, 16, 4, 64, 1, nul, nul) == L.PA_OK
    assert lib.pa_copy_blocks(nul, nul, nul, 2, 64, 16, 4, 64, 1, nul, nul) == L.PA_ERR_INVALID_ARG
    misaligned = ctypes.c_void_p(0x1008)
    assert lib.pa_copy_blocks(misaligned, misaligned, misaligned, 2, 64, 16, 4, 64, 1, nul, nul) == \
        L.PA_ERR_INVALID_ARG


def declared_prototypes():
    """{name: (return type, [parameter types])} from include/*.h, comments removed."""
    protos = {}
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = "\n".join(line for line in src.splitlines() if not line.lstrip().startswith("#"))
        for m in re.finditer(r"([A-Za-z_][\w\s\*]*?)\b(pa_\w+)\s*\(([^;{]*?)\)\s*;", src):
            ret, name, params = " ".join(m.group(1).split()), m.group(2), m.group(3)
            params = [" ".join(p.split()) for p in params.split(",")] if params.strip() not in ("", "void") else []
            protos[name] = (ret, params)
    return protos


def _ctype_of(decl: str):
    if "*" in decl:
        return ctypes.c_char_p if decl.startswith("const char") else ctypes.c_void_p
    base = decl.split()[0] if decl.split()[0] != "const" else decl.split()[1]
    return {"int": ctypes.c_int, "int32_t": ctypes.c_int, "pa_status": ctypes.c_int, "pa_dtype": ctypes.c_int,
            "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t, "float": ctypes.c_float}[base]


def test_binding_signatures_match_the_header():
    """Every ctypes signature has the header prototype's arity and types, so
    no argument is shifted or truncated on the way into the library."""
    from paged_kv_cache_140_gb300 import _lib
    protos = declared_prototypes()
    assert set(protos) == set(declared_functions())
    for name, (ret, params) in protos.items():
        res, args = _lib.SIGNATURES[name]
        assert len(args) == len(params), f"{name}: {len(args)} bound, {len(params)} declared"
        for i, (a, decl) in enumerate(zip(args, params)):
            want = _ctype_of(decl)
            pointer_ok = want is ctypes.c_void_p and issubclass(a, ctypes._Pointer)
            assert a is want or pointer_ok, f"{name} argument {i} ({decl}): bound as {a.__name__}"
        want = _ctype_of(ret + (" *" if ret.endswith("*") else ""))
        assert res is want or (res is ctypes.c_int and want is ctypes.c_int), f"{name} returns {ret}"
