"""The C-ABI library loads and exports every function the headers declare (no GPU).

Only symbol lookup happens here; no call that touches a device is made.
"""
import ctypes
import os
import re

from step_gpt_train_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DECL = re.compile(r"^\s*(?:const\s+)?(?:int|int64_t|size_t|char\s*\*|void)\s*\**\s*(gpt2_\w+)\s*\(", re.M)


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            names |= set(DECL.findall(open(os.path.join(inc, f)).read()))
    return names


def test_headers_declare_the_step_calls():
    names = declared_functions()
    for n in ("gpt2_init", "gpt2_forward", "gpt2_backward", "gpt2_adamw_step"):
        assert n in names
    assert len(names) >= 30


def test_library_exports_every_declared_symbol():
    path = _build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in sorted(declared_functions()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from step_gpt_train_gb300 import gpt2 as g
    missing = sorted(declared_functions() - set(g._SIGNATURES))
    assert not missing, missing
    g.load_library()  # sets every argtype; raises if a name is absent


def test_library_needs_no_driver_library():
    # the CUDA runtime is linked statically and the driver entry point is looked
    # up at run time, so the library's dynamic dependencies name no CUDA library
    import shutil
    import subprocess
    import pytest
    if not shutil.which("readelf"):
        pytest.skip("readelf not available")
    path = _build.build()
    out = subprocess.run(["readelf", "-d", path], capture_output=True, text=True).stdout
    needed = [l for l in out.splitlines() if "(NEEDED)" in l]
    assert needed and not any("libcuda" in l or "libcudart" in l for l in needed), needed


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback: without the built library every entry point of the binding raises
    import pytest
    from step_gpt_train_gb300 import gpt2 as g
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g._build, "LIB", str(tmp_path / "absent" / "libgpt2.so"))
    with pytest.raises(ImportError):
        g.load_library()
    with pytest.raises(ImportError):
        g.gpt2_lr_cosine(1, 1, 10, 1e-3, 0.0)
