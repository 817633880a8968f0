import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_available():
    import torch
    return torch.cuda.is_available()


def pytest_terminal_summary(terminalreporter):
    """The parity record of the GPU tests: steps compared against the oracle,
    and those whose binary32 clip coefficient differed from the oracle's (from
    such a step on the elements were held to the tolerance, not to bit
    identity)."""
    gc = sys.modules.get("gpu_common")
    if gc is not None and gc.Parity.steps:
        terminalreporter.write_line(
            f"parity: {gc.Parity.steps} applied steps compared with the oracle; "
            f"clip coefficient differed in {gc.Parity.clip_differs}; "
            f"of {gc.Parity.bounded} elements compared under a derived bound after such a step, "
            f"{gc.Parity.tight} were beyond 1e-6 rel + 1e-12 abs (and within the bound)")
