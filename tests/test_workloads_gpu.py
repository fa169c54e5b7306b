"""Parity at the full sizes of the measured workloads, in the launch configurations the
benchmark times.  The GPU always runs the whole workload; the fp64 oracle checks a sample of
(sequence, v-head) pairs, or the whole result where that is cheap.

  * varlen layer: 64 replay tails of one layer (lengths drawn from the seed), bf16.
  * full 32K: one 32768-token sequence, bf16 (the replay-vs-full comparison's full side).
  * chunk operators of 16 isolated 2048-token chunks, 32 v-heads, fp32, with the config's
    gates (T_C underflows to zero) and with weak-decay gates (T_C non-trivial).
  * composition of those 16 operators (K = 16, 32 heads, d = 128), fp32.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_state_chunked_gb300 import _lib, api, synthetic
from tests.gpu_util import TOL_BF16, TOL_F32, host, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    _lib.load(build=True)
    torch.cuda.init()


def _sampled_replay_check(x, O, S, pairs, tol):
    S_ref, O_ref = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.S0, sel=pairs)
    Sg, Og = host(S), host(O)
    cu = x.cu_seqlens
    for seq, h in pairs:
        es = rel_err(Sg[seq, h], S_ref[seq, h])
        rows = slice(int(cu[seq]), int(cu[seq + 1]))
        eo = rel_err(Og[rows, h], O_ref[rows, h])
        assert es <= tol and eo <= tol, f"(seq {seq}, head {h}): S {es:.3e}, O {eo:.3e}"


def test_varlen_layer_sampled():
    x = synthetic.varlen_workload_inputs(0)
    d = to_device(x)
    O, S = api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    torch.cuda.synchronize()
    api.gdn_get_status()
    lengths = np.diff(x.cu_seqlens)
    longest, shortest = int(np.argmax(lengths)), int(np.argmin(lengths))
    pairs = [(longest, 0), (longest, 31), (shortest, 5), (17, 12), (40, 19), (63, 30)]
    _sampled_replay_check(x, O, S, pairs, TOL_BF16)


def test_full_32k_sampled():
    x = synthetic.workload_inputs("full_32k")
    d = to_device(x)
    O, S = api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    torch.cuda.synchronize()
    api.gdn_get_status()
    _sampled_replay_check(x, O, S, [(0, 0), (0, 21)], TOL_BF16)


@pytest.mark.parametrize("weak_decay", [False, True])
def test_chunk_operators_and_composition(weak_decay):
    x = synthetic.chunk_workload_inputs(weak_decay=weak_decay)
    d = to_device(x)
    K = len(x.cu_seqlens) - 1
    T, Sl = api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu_seqlens"])
    SK = api.gdn_compose([T[j] for j in range(K)], [Sl[j] for j in range(K)])
    torch.cuda.synchronize()
    api.gdn_get_status()
    Tg, Slg, SKg = host(T), host(Sl), host(SK)
    # oracle operators for v-heads 0, 1 (key head 0) and 30, 31 (key head 15)
    vh, kh = [0, 1, 30, 31], [0, 15]
    T_ref, Sl_ref = oracle.chunk_operator(x.k[:, kh], x.g[:, vh], x.beta[:, vh], x.v[:, vh], x.cu_seqlens)
    assert rel_err(Slg[:, vh], Sl_ref) <= TOL_F32
    if weak_decay:
        assert rel_err(Tg[:, vh], T_ref) <= TOL_F32
    else:
        # the config's gates sum to about -436 over a chunk: T_C is below the fp32 range
        assert np.abs(Tg[:, vh] - T_ref).max() <= 1e-30
    # composition: all heads against the closed form of the GPU's own operators, and the
    # sampled heads against the closed form of the oracle's operators
    assert rel_err(SKg, oracle.compose(Tg, Slg)) <= TOL_F32
    assert rel_err(SKg[vh], oracle.compose(T_ref, Sl_ref)) <= TOL_F32
