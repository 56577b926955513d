"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the built CUDA library; the rest
run on a CPU-only machine.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


def read_golden(name):
    """Parse a `key = values` fixture file into a dict of float lists (or strings)."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or "=" not in line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = [float(t) for t in v.split()]
    return out


def read_masks(name):
    """Parse the causal-mask fixture into {(Nq, Nk): [[0/1...]...]}."""
    masks, cur = {}, None
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("mask"):
                kv = dict(t.split("=") for t in line.split()[1:])
                cur = (int(kv["seqlen_q"]), int(kv["seqlen_k"]))
                masks[cur] = []
            else:
                masks[cur].append([int(t) for t in line.split()])
    return masks


@pytest.fixture(scope="session")
def golden_example():
    return read_golden("worked_example.txt")


@pytest.fixture(scope="session")
def golden_masks():
    return read_masks("causal_masks.txt")
