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


def check_steps(got, got_am, ref, rel_tol=2e-2):
    """Per-step logits and argmax of a decode run against the oracle's rows.

    Every step: max |got - ref| <= rel_tol * std(ref), and the device's argmax
    is the argmax of its own logits.  Where that token differs from the
    oracle's argmax, the oracle must rate it within twice the step's measured
    logit error of its maximum (a tie at the precision both sides reach; no
    step is exempt).  Returns the number of such steps, which callers bound."""
    diff = 0
    for i in range(ref.shape[0]):
        err = float(np.abs(got[i] - ref[i]).max())
        tol = rel_tol * ref[i].std()
        assert err <= tol, (i, err, tol)
        assert got_am[i] == int(np.argmax(got[i])), i
        best = int(np.argmax(ref[i]))
        if got_am[i] != best:
            diff += 1
            assert ref[i][got_am[i]] >= ref[i][best] - 2 * err, (i, ref[i][best] - ref[i][got_am[i]], err)
    return diff
