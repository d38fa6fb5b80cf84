import os
import sys

# Bounded device waits give up after 1 s in tests (a legitimate wait takes
# microseconds), so a protocol bug surfaces as a reported timeout quickly.
os.environ.setdefault("CPATTN_WAIT_LIMIT_MS", "1000")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
