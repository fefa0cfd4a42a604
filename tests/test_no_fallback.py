"""The product path has no CPU fallback (CPU only).

With the CUDA library absent every entry of the binding raises before doing
any work; nothing in the package imports the oracle, and the oracle imports
nothing from the package and includes only system headers.
"""
import ast
import glob
import os

import pytest
import torch

from bit_fp8_attention_means_gb300 import vc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture
def no_library(monkeypatch, tmp_path):
    monkeypatch.setattr(vc, "_lib", None)
    monkeypatch.setattr(vc, "LIB_PATH", str(tmp_path / "libvc_gb300.so"))
    yield


def test_every_call_raises_without_the_library(no_library):
    x = torch.zeros((1, 256, 2, 64), dtype=torch.bfloat16)
    s = vc.shape_of(x)
    with pytest.raises(RuntimeError, match="libvc_gb300.so is missing"):
        vc.lib()
    for call in (lambda: vc.vc_cluster(x, 4, 1),
                 lambda: vc.vc_quantize(x, x, x, None, 1),
                 lambda: vc.vc_quantize_ex(x, x, x, None, 1, hadamard=1)):
        with pytest.raises(RuntimeError, match="libvc_gb300.so is missing"):
            call()
    # the attention call asks for the current CUDA stream first: on a machine
    # without a GPU that raises too; either way nothing runs on the host
    with pytest.raises(RuntimeError):
        vc.vc_attn_fwd(vc.alloc_quantized(s, x.device, 1), s)


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(ROOT, "bit_fp8_attention_means_gb300", "*.py")):
        tree = ast.parse(open(path).read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            else:
                continue
            assert not any(n == "oracle" or n.startswith("oracle.") for n in names), (path, names)


def test_oracle_shares_no_code_with_the_library():
    """The oracle imports nothing from the package and includes only system headers."""
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        tree = ast.parse(open(path).read())
        for node in ast.walk(tree):
            if isinstance(node, (ast.Import, ast.ImportFrom)):
                names = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
                assert not any(n.startswith("bit_fp8_attention_means_gb300") for n in names), (path, names)
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.c")):
        for line in open(path):
            if line.lstrip().startswith("#include"):
                assert "<" in line and '"' not in line, (path, line)
