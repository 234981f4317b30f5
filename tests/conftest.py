"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the compiled sm_103a library; the
rest run on any CPU.  The repository root is put on ``sys.path`` so that the
``oracle`` test package and ``paged_attention_decode_gb300`` import without
installation.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the compiled library")
