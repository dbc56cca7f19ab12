"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on a CPU-only machine.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled fhd library")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")
    config.addinivalue_line("markers", "auto_path: GPU parity test that keeps the library's automatic path choice")
