import ast
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def load_golden(name):
    """Parse tests/golden/<name>: `key = <python literal>` lines, '#' comments."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    buf = ""
    with open(path, encoding="utf-8") as f:
        for line in f:
            s = line.strip()
            if not s or s.startswith("#"):
                continue
            buf = (buf + " " + s) if buf else s
            key, _, val = buf.partition("=")
            try:
                out[key.strip()] = ast.literal_eval(val.strip())
                buf = ""
            except SyntaxError:
                continue  # value spans several lines
    assert not buf, f"unterminated golden entry: {buf[:60]}"
    return out


@pytest.fixture(scope="session")
def page():
    return load_golden("page_layouts.txt")
