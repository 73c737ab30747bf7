"""The C-ABI library builds, loads and exports every entry point that
include/easyspec.h declares (no compute calls: runs without a GPU)."""
import os
import re
import subprocess

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "easyspec.h")


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"ES_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ("easyspec_init", "draft_step", "verify_step", "calibrate_kv", "generate",
                 "es_accept_resample", "easyspec_destroy", "easyspec_last_error"):
        assert must in names


def test_library_builds_and_exports_every_declared_symbol():
    from layer_drafting_draft_b300 import build, easyspec
    path = build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    L = easyspec.lib()  # dlopen works without a GPU
    for n in declared_symbols():
        assert hasattr(L, n)
    assert sorted(easyspec.EXPORTED) == declared_symbols()


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from layer_drafting_draft_b300 import easyspec
    monkeypatch.setattr(easyspec, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(easyspec, "_lib", None)
    import pytest
    with pytest.raises(RuntimeError, match="missing"):
        easyspec.lib()
