"""Helpers of the GPU parity tests: move seeded inputs to the device, run the oracle."""
import numpy as np
import torch

import oracle

TOL_F32 = 1e-5   # relative Frobenius, fp32 inputs (fp32 CUDA-core path)
TOL_BF16 = 3e-3  # relative Frobenius, bf16 inputs with fp32 accumulation


def to_device(x, dev="cuda"):
    """ReplayInputs -> dict of device tensors (bf16 values are exact copies)."""
    dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32

    def t(a, d):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev).to(d)

    out = dict(q=t(x.q, dt), k=t(x.k, dt), v=t(x.v, dt), g=t(x.g, torch.float32), beta=t(x.beta, torch.float32),
               cu_seqlens=t(x.cu_seqlens, torch.int32))
    out["S0"] = None if x.S0 is None else t(x.S0, torch.float32)
    return out


def oracle_replay(x, l2norm_qk=True, scale=1.0, want_O=True, sel=None, scalar_decay=False):
    return oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.S0, l2norm_qk=l2norm_qk, scale=scale,
                         want_O=want_O, sel=sel, scalar_decay=scalar_decay)


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


rel_err = oracle.rel_err
