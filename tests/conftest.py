import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU with the sm_103a library built")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_terminal_summary(terminalreporter):
    """Near-tie selections the oracle adopted from the GPU, per parity comparison."""
    mod = sys.modules.get("_gpu")
    log = getattr(mod, "FLAG_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tr.section("oracle follow mode: near-tie selections adopted per comparison")
    total = 0
    for test, cfg, n, flags, gap in log:
        total += flags
        tr.write_line(f"{flags:4d} flags  max gap {gap:.2e}  {n:3d} request(s)  {cfg:22s} {test}")
    tr.write_line(f"{total} adopted near-tie selection(s) in {len(log)} comparison(s)")
