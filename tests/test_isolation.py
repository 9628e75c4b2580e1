"""The oracle and the CUDA path share no code, and the product never reaches
the oracle: importing the package loads no oracle module, no product source
names it, and the oracle includes or imports nothing of the package (the
seeded input generator, which holds none of the method's arithmetic, is
passed to it as data by the tests)."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_140_gb300")


def _files(top, exts):
    for d, _, fs in os.walk(top):
        if "__pycache__" in d or os.sep + "_build" in d or os.sep + "lib" in d[len(top):]:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_importing_the_package_loads_no_oracle():
    code = ("import sys; import paged_kv_cache_140_gb300 as pa; import paged_kv_cache_140_gb300._lib; "
            "import paged_kv_cache_140_gb300.workloads; "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "print(bad); sys.exit(1 if bad else 0)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr


def test_no_product_source_refers_to_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|#\s*include\s*[<\"][^>\"]*oracle)", re.M)
    for f in _files(PKG, (".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
        assert not pat.search(open(f, encoding="utf-8").read()), f
    for f in _files(os.path.join(ROOT, "include"), (".h",)):
        assert not pat.search(open(f, encoding="utf-8").read()), f


def test_oracle_uses_nothing_of_the_cuda_path():
    inc = re.compile(r"^\s*#\s*include\s*\"", re.M)                       # only system headers
    imp = re.compile(r"^\s*(import|from)\s+paged_kv_cache_140_gb300", re.M)
    for f in _files(os.path.join(ROOT, "oracle"), (".c", ".h", ".cpp")):
        assert not inc.search(open(f, encoding="utf-8").read()), f
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        assert not imp.search(open(f, encoding="utf-8").read()), f


def test_missing_library_fails_loudly():
    """Without the built CUDA library a call raises; there is no fallback."""
    code = ("import sys, paged_kv_cache_140_gb300._lib as L, paged_kv_cache_140_gb300._build as B; "
            "B.LIB_PATH = '/nonexistent/libpagedattn.so'; L._lib = None\n"
            "try:\n    L.load()\nexcept ImportError as e:\n    print('raised', e); sys.exit(0)\nsys.exit(1)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "is missing" in r.stdout, r.stdout + r.stderr
