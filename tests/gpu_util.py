"""Helpers for the GPU parity tests: device upload and download."""
import numpy as np
import torch


def dev():
    return torch.device("cuda:0")


def up(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def down(t) -> np.ndarray:
    return t.cpu().numpy()
