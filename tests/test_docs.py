"""The Python example of README.md is valid Python and calls only names the
binding defines (it was run on a B300; here it is checked without a GPU)."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_uses_binding_names():
    from nvfp4_precision_02_b300 import binding
    text = open(os.path.join(ROOT, "README.md")).read()
    sec = text[text.index("## Python\n"):text.index("## C\n")]
    code = "\n".join(l[4:] for l in sec.splitlines() if l.startswith("    "))
    tree = ast.parse(code)
    used = {n.attr for n in ast.walk(tree)
            if isinstance(n, ast.Attribute) and isinstance(n.value, ast.Name) and n.value.id == "nv"}
    assert {"quantize_1d", "quantize_2d", "gemm", "SR"} <= used
    for name in used:
        assert hasattr(binding, name), name
