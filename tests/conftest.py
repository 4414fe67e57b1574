import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


# Runs against the bounds-checked debug build (SPEC_VERIFY_LIBRARY names it):
# after every GPU test, no index check of the library may have failed.
if os.environ.get("SPEC_VERIFY_LIBRARY"):
    import pytest

    @pytest.fixture(autouse=True)
    def _no_debug_flags(request):
        yield
        if request.node.get_closest_marker("gpu") is None:
            return
        from draft_token_verification_sv_gb300 import _native as N
        if N._lib is None:
            return
        assert N.LIB_PATH == os.environ["SPEC_VERIFY_LIBRARY"]
        flags = N.lib().sv_debug_flags(1)
        assert flags == 0, f"bounds checks of the debug build failed: flags {flags:#x}"
