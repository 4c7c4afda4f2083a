"""The Python example (examples/fprop_dgrad.py) is valid Python and calls
only names the binding defines (here it is checked without a GPU)."""
import ast
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_python_example_uses_binding_names():
    from nvfp4_precision_02_b300 import binding
    code = open(os.path.join(ROOT, "examples", "fprop_dgrad.py")).read()
    tree = ast.parse(code)
    used = {n.attr for n in ast.walk(tree)
            if isinstance(n, ast.Attribute) and isinstance(n.value, ast.Name) and n.value.id == "nv"}
    assert {"quantize_1d", "quantize_2d", "gemm", "SR"} <= used
    for name in used:
        assert hasattr(binding, name), name


@pytest.mark.gpu
def test_python_example_runs():
    """The Python example runs end to end on the GPU."""
    import importlib.util
    import torch
    assert torch.cuda.is_available()
    spec = importlib.util.spec_from_file_location("fprop_dgrad", os.path.join(ROOT, "examples", "fprop_dgrad.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.main()
    from nvfp4_precision_02_b300 import binding
    assert binding.device_status() == 0
