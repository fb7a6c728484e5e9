"""Shared pytest setup: repository root on sys.path and the `gpu` marker.

Tests marked `gpu` need a CUDA device and the compiled library; everything else runs on CPU.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")
