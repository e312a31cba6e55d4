"""The Python binding on the host (no GPU): it refuses host tensors instead of computing on
the CPU, raises when the compiled library is missing, and the product package and the
oracle never import one another."""
import ast
import os

import pytest
import torch

import convolution_nchw_conv2d_gb300 as cg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "convolution_nchw_conv2d_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _host_calls():
    x = torch.ones(1, 2, 5, 5)
    w = torch.ones(3, 2, 3, 3)
    dy = torch.ones(1, 3, 3, 3)
    x1 = torch.ones(1, 2, 5)
    w1 = torch.ones(3, 2, 3)
    dy1 = torch.ones(1, 3, 3)
    x3 = torch.ones(1, 2, 4, 5, 5)
    w3 = torch.ones(3, 2, 2, 3, 3)
    dy3 = torch.ones(1, 3, 3, 3, 3)
    return {
        "conv2d_fwd": lambda: cg.conv2d_fwd(x, w),
        "conv2d_fwd_noalloc": lambda: cg.conv2d_fwd_noalloc(x, w),
        "conv2d_bwd_data": lambda: cg.conv2d_bwd_data(dy, w, (5, 5)),
        "conv2d_bwd_filter": lambda: cg.conv2d_bwd_filter(x, dy, (3, 3)),
        "deconv2d_fwd": lambda: cg.deconv2d_fwd(dy, w, (5, 5)),
        "conv1d_fwd": lambda: cg.conv1d_fwd(x1, w1),
        "conv1d_bwd_data": lambda: cg.conv1d_bwd_data(dy1, w1, 5),
        "conv1d_bwd_filter": lambda: cg.conv1d_bwd_filter(x1, dy1, 3),
        "conv2d_bwd": lambda: cg.conv2d_bwd(x, w, dy),
        "conv3d_fwd": lambda: cg.conv3d_fwd(x3, w3),
        "conv3d_bwd_data": lambda: cg.conv3d_bwd_data(dy3, w3, (4, 5, 5)),
        "conv3d_bwd_filter": lambda: cg.conv3d_bwd_filter(x3, dy3, (2, 3, 3)),
    }


@pytest.mark.parametrize("name", sorted(_host_calls()))
def test_host_tensors_are_refused(name):
    """Every compute entry point rejects host tensors: there is no CPU path to fall back on."""
    with pytest.raises(ValueError, match="CUDA tensor"):
        _host_calls()[name]()


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(cg, "_lib", None)
    monkeypatch.setattr(cg, "_LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        cg.load_library()
    with pytest.raises(RuntimeError, match="missing"):
        cg.conv2d_output_dim(8, 1, 3, 1)


def _imported_modules(folder):
    names = set()
    for dirpath, _, files in os.walk(folder):
        for f in files:
            if not f.endswith(".py"):
                continue
            tree = ast.parse(open(os.path.join(dirpath, f)).read())
            for node in ast.walk(tree):
                if isinstance(node, ast.Import):
                    names.update(a.name.split(".")[0] for a in node.names)
                elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
                    names.add(node.module.split(".")[0])
    return names


def test_product_and_oracle_do_not_import_each_other():
    assert "oracle" not in _imported_modules(PKG)
    assert "convolution_nchw_conv2d_gb300" not in _imported_modules(ORACLE)


def test_product_sources_name_no_oracle_file():
    """Neither the CUDA sources nor the binding include, load or open a file of the oracle."""
    artifacts = sorted(f for f in os.listdir(ORACLE) if f.endswith((".c", ".py"))) + ["liboracle", "oracle/"]
    for dirpath, _, files in os.walk(PKG):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                for a in artifacts:
                    if a == "__init__.py":
                        continue
                    assert a not in text, (f, a)
