"""Test helper: build (if stale) and load the library; skip GPU tests without a GPU."""
import torch

from reproducible_deterministic_attn_gb300 import build as _build


def ensure_built():
    _build.build()


def has_gpu() -> bool:
    return torch.cuda.is_available()
