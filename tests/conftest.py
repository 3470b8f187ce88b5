import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpkv")
    config.addinivalue_line("markers", "slow: full-size parity cases")


@pytest.fixture(autouse=True)
def _reload_tuning_after_test():
    # a test may change PKV_ATTN_* tuning variables (through helpers.set_knobs);
    # once its monkeypatch has restored the environment, the library re-reads them
    yield
    mod = sys.modules.get("paged_kv_cache_243_gb300.binding")
    if mod is not None and getattr(mod, "_lib", None) is not None:
        mod.tuning_reload()
