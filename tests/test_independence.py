"""The oracle and the CUDA path share no code: a static check of the sources.

The package (its binding, build script, workload generators and CUDA/C++
sources) never imports, loads or includes anything under oracle/, and the
oracle imports nothing from the package and includes none of its headers.
"""
import pathlib
import re

ROOT = pathlib.Path(__file__).resolve().parents[1]
PKG = ROOT / "prefix_tree_block_gb300"
ORACLE = ROOT / "oracle"


def _sources(d, exts):
    return [p for p in d.rglob("*") if p.suffix in exts and "_build" not in p.parts]


def test_package_does_not_reach_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"][^>\"]*oracle)|oracle\.(c|so|py)\b|"
                     r"liboracle", re.M)
    for p in _sources(PKG, {".py", ".cu", ".cuh", ".h", ".cpp", ".c"}) + list((ROOT / "include").glob("*.h")):
        hits = pat.findall(p.read_text())
        assert not hits, f"{p.relative_to(ROOT)} refers to the oracle: {hits}"


def test_oracle_does_not_reach_the_package():
    pat = re.compile(r"prefix_tree_block_gb300|libpt|#\s*include\s*\"(pt|pt_[a-z_]+)\.(h|cuh)\"")
    for p in _sources(ORACLE, {".py", ".c", ".h"}):
        hits = pat.findall(p.read_text())
        assert not hits, f"{p.relative_to(ROOT)} refers to the CUDA path: {hits}"
