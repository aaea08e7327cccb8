"""Static checks on the product sources: the library's Python binding and layer harness never reach the
FP64 oracle (it is test infrastructure), and the CUDA sources hold no deliberate trap (every wait in the
kernels is bounded and reports an error status instead)."""
import pathlib
import re

ROOT = pathlib.Path(__file__).resolve().parents[1]
PKG = ROOT / "linear_attention_mixer_gb300"


def _product_python():
    return sorted(PKG.glob("*.py"))


def _cuda_sources():
    csrc = PKG / "csrc"
    return sorted(list(csrc.glob("*.cu")) + list(csrc.glob("*.cuh")) + list((ROOT / "include").glob("*.h")))


def test_product_python_does_not_import_the_oracle():
    files = _product_python()
    assert files
    for p in files:
        src = p.read_text()
        assert not re.search(r"^\s*(from\s+oracle\b|import\s+oracle\b)", src, re.M), p.name
        assert "oracle." not in re.sub(r"#.*", "", src), p.name


def test_cuda_sources_have_no_trap():
    files = _cuda_sources()
    assert files
    for p in files:
        src = p.read_text()
        assert "__trap" not in src, p.name
        assert not re.search(r"\btrap\s*;", src), p.name
        assert "__brkpt" not in src, p.name
