"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import oracle
import synth
from weight_only_quantized_bs_gb300.weights import to_dev


def bf16_host(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def as_f64(t):
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_double(bf16_host(t))
    return t.detach().cpu().double().numpy()


def rel_err(y, ref):
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


def weights(N, K, tid, seed=0):
    return synth.normal_bf16(seed, tid, (N, K), 0.02)


def xvec(K, tid, seed=0):
    return synth.normal_bf16(seed, tid, (K,), 1.0)


__all__ = ["bf16_host", "as_f64", "rel_err", "weights", "xvec", "to_dev"]
