"""Helpers shared by the GPU parity tests: device copies to numpy bit patterns and a
lazy per-expert weight accessor for the oracle (one expert copied to the host at a time)."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bits(t):
    """BF16 (or int16) tensor -> numpy uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    return t.detach().cpu().numpy()


class ExpertBits:
    """Indexable view of a [E, ...] BF16 device tensor: [e] -> numpy uint16 bits of expert e."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return bits(self.t[int(e)])


def sample_tokens(T_valid, n, seed=0):
    rng = np.random.default_rng(seed)
    if n >= T_valid:
        return np.arange(T_valid)
    picks = rng.choice(T_valid, size=n, replace=False)
    return np.unique(np.concatenate([picks, [0, T_valid - 1]]))
