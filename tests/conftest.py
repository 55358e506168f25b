import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

# Temporary files of the tests (compiled oracle mutants, C test programs) stay
# inside the repository, under a git-ignored folder.
os.environ.setdefault("PYTEST_DEBUG_TEMPROOT", os.path.join(ROOT, ".pytest_tmp"))
os.makedirs(os.environ["PYTEST_DEBUG_TEMPROOT"], exist_ok=True)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
