import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The readout tolerance's bookkeeping: how many bf16 readouts the GPU parity tests
    compared with the oracle and how many passed only by the cancellation rule (ii)."""
    mod = sys.modules.get("parity_util")
    R = getattr(mod, "READOUT_REPORT", None)
    if R and R["readouts"]:
        terminalreporter.write_line(
            f"readouts compared with the oracle: {R['readouts']}; worst distance "
            f"{R['worst_ulp']} bf16 steps; passed only by the cancellation rule: "
            f"{R['rule_ii']} (worst |err|/bound {R['rule_ii_worst_frac']:.3f}, largest "
            f"|y|/sum|S'C| among them {R['rule_ii_least_cancellation']:.2e})")
