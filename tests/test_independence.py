"""The product path and the oracle share nothing: no file of the package
(binding, build script, CUDA sources) imports, includes or names a module of
oracle/, and oracle/ imports nothing of the package.  The package builds
for sm_103a only.  CPU only."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mtp_self_speculative_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d or "_build" in os.path.relpath(d, top).split(os.sep)[0:1]:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_does_not_reach_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|#\s*include\s+[\"<][^\">]*oracle)", re.M)
    hits = [p for p in _files(PKG, (".py", ".cu", ".cuh", ".h")) if pat.search(open(p, encoding="utf-8").read())]
    assert not hits, hits


def test_oracle_does_not_reach_the_package():
    pat = re.compile(r"^\s*(import|from)\s+mtp_self_speculative_gb300\b", re.M)
    hits = [p for p in _files(os.path.join(ROOT, "oracle"), (".py",)) if pat.search(open(p, encoding="utf-8").read())]
    assert not hits, hits


def test_build_targets_sm_103a_only():
    src = open(os.path.join(PKG, "_build.py"), encoding="utf-8").read()
    arches = re.findall(r"arch=compute_(\w+),code=sm_(\w+)", src)
    assert arches == [("103a", "103a")], arches
