"""GPU parity of the tensor-core path (bf16 inputs, d_k = d_v = 128) against the fp64 oracle.

gdn_replay takes this path for bf16 inputs unless GDN_PRECISE is set.  The
bar is a relative Frobenius error <= 3e-3 on S and O (bf16 inputs, fp32
accumulation and state, O rounded to bf16).  Cases span several chunks,
ragged tails (partial last chunks, one-token and empty tails), both state
slicings (32-row slices for few problems, 64-row slices for many), an
entering state, the in-kernel q/k normalisation on raw inputs, a non-unit
readout scale, weak-decay gates that make the chunk-to-chunk carry matter,
and the full single-layer workloads (3277- and 1638-token tails, 16 q/k heads
shared by 32 v heads).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_state_chunked_gb300 import _lib, api, synthetic
from tests.gpu_util import TOL_BF16, host, oracle_replay, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    _lib.load(build=True)
    torch.cuda.init()


def _run(x, **kw):
    d = to_device(x)
    O, S = api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["S0"], **kw)
    torch.cuda.synchronize()
    api.gdn_get_status()
    return O, S


def _check(x, O, S, tol=TOL_BF16, **kw):
    S_ref, O_ref = oracle_replay(x, **kw)
    es = rel_err(host(S), S_ref)
    assert es <= tol, f"S rel err {es:.3e}"
    if O is not None:
        eo = rel_err(host(O), O_ref)
        assert eo <= tol, f"O rel err {eo:.3e}"
        return es, eo
    return es, None


@pytest.mark.parametrize("name", ["layer_r1638", "layer_r3277"])
def test_single_layer_workload(name):
    x = synthetic.workload_inputs(name)
    O, S = _run(x)
    _check(x, O, S)


RAGGED = [1, 63, 64, 65, 130, 0, 200]


@pytest.mark.parametrize("with_S0", [False, True])
def test_ragged_few_problems_32_row_slices(with_S0):
    assert _lib.load() and api  # library present
    x = synthetic.make_replay_inputs(RAGGED, 2, 4, 128, 128, dtype="bf16", seed=300 + with_S0, unit_qk=False,
                                     with_S0=with_S0)
    O, S = _run(x, scale=0.5)
    _check(x, O, S, scale=0.5)


def test_ragged_many_problems_64_row_slices():
    rng = np.random.Generator(np.random.PCG64(301))
    lengths = [int(v) for v in rng.integers(0, 300, size=24)]
    x = synthetic.make_replay_inputs(lengths, 2, 4, 128, 128, dtype="bf16", seed=302, with_S0=True)
    O, S = _run(x)
    _check(x, O, S)


def test_many_tails_each_replayed_once():
    """300 tails (more than one block of the longest-first ordering), lengths out of order and
    with ties, so that the scan's grid takes them in a permuted order: every tail's state must
    match the oracle on its own (a tail skipped or taken twice would not)."""
    rng = np.random.Generator(np.random.PCG64(310))
    lengths = [int(v) for v in rng.integers(0, 140, size=290)] + [70] * 10
    rng.shuffle(lengths)
    x = synthetic.make_replay_inputs(lengths, 1, 2, 128, 128, dtype="bf16", seed=311, with_S0=True)
    O, S = _run(x)
    S_ref, O_ref = oracle_replay(x)
    Sh = host(S)
    worst = max(rel_err(Sh[i], S_ref[i]) for i in range(len(lengths)))
    assert worst <= TOL_BF16, f"worst per-tail S rel err {worst:.3e}"
    assert rel_err(host(O), O_ref) <= TOL_BF16


@pytest.mark.parametrize("h_k,h_v", [(1, 4), (1, 3)])
def test_more_than_two_v_heads_per_key_head(h_k, h_v):
    """Four and three v-heads per key head: the prep kernel treats a key head's v-heads in
    pairs, so these take its second pass (and an odd last pair)."""
    x = synthetic.make_replay_inputs([130, 64, 5], h_k, h_v, 128, 128, dtype="bf16", seed=320 + h_v,
                                     with_S0=True)
    O, S = _run(x)
    _check(x, O, S)


def test_weak_decay_carry():
    """g scaled by 1e-3: the state entering each chunk dominates, so errors in the
    inter-chunk carry would show."""
    x = synthetic.make_replay_inputs([1000, 333], 2, 4, 128, 128, dtype="bf16", seed=303, gate_scale=1e-3,
                                     with_S0=True)
    O, S = _run(x)
    _check(x, O, S)


def test_without_l2norm():
    x = synthetic.make_replay_inputs([150, 77], 2, 4, 128, 128, dtype="bf16", seed=304)
    O, S = _run(x, l2norm_qk=False)
    _check(x, O, S, l2norm_qk=False)


def test_state_only():
    x = synthetic.make_replay_inputs([500, 64, 3], 2, 4, 128, 128, dtype="bf16", seed=305, with_S0=True)
    _, S = _run(x, state_only=True)
    _check(x, None, S, want_O=False)


def test_matches_precise_path():
    """The tensor-core path and the fp32 CUDA-core path agree to the bf16 bar."""
    x = synthetic.make_replay_inputs([260, 31], 2, 4, 128, 128, dtype="bf16", seed=306, with_S0=True)
    O1, S1 = _run(x)
    O2, S2 = _run(x, precise=True)
    assert rel_err(host(S1), host(S2)) <= TOL_BF16
    assert rel_err(host(O1), host(O2)) <= TOL_BF16


def test_rows_outside_sequences_untouched():
    x = synthetic.make_replay_inputs([100, 40], 2, 4, 128, 128, dtype="bf16", seed=307)
    d = to_device(x)
    cu = torch.tensor([0, 100, 120], dtype=torch.int32, device="cuda")
    O = torch.full((140, 4, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, O_out=O)
    torch.cuda.synchronize()
    assert torch.all(O[120:] == 3.0)
    S_ref, O_ref = oracle.replay(x.q, x.k, x.v, x.g, x.beta, [0, 100, 120])
    assert rel_err(host(O[:120]), O_ref[:120]) <= TOL_BF16


@pytest.mark.parametrize("state_only", [True, False])  # the operator-form scan / the scan with outputs
def test_malformed_cu_seqlens_reports_shape_error(state_only):
    x = synthetic.make_replay_inputs([64, 64], 2, 4, 128, 128, dtype="bf16", seed=308)
    d = to_device(x)
    cu = torch.tensor([0, 100, 50], dtype=torch.int32, device="cuda")
    S = torch.full((2, 4, 128, 128), 9.0, device="cuda")
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S_out=S, state_only=state_only)
    with pytest.raises(_lib.GdnError) as ei:
        api.gdn_get_status()
    assert ei.value.code == _lib.GDN_ERR_SHAPE
    assert torch.all(S[1] == 9.0)


@pytest.mark.parametrize("state_only", [True, False])
def test_overlapping_forward_ranges_report_shape_error(state_only):
    """Offsets that each run forward but go back ([0, T, 0, T]) would hold more chunks than the
    per-chunk buffers: the ranges after the step back are skipped and reported, nothing else."""
    T = 200
    x = synthetic.make_replay_inputs([T], 2, 4, 128, 128, dtype="bf16", seed=310)
    d = to_device(x)
    cu = torch.tensor([0, T, 0, T], dtype=torch.int32, device="cuda")
    S = torch.full((3, 4, 128, 128), 7.0, device="cuda")
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S_out=S, state_only=state_only)
    with pytest.raises(_lib.GdnError) as ei:
        api.gdn_get_status()
    assert ei.value.code == _lib.GDN_ERR_SHAPE
    assert torch.all(S[1] == 7.0) and torch.all(S[2] == 7.0)
    S_ref, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, [0, T], want_O=False)
    assert rel_err(host(S[0]), S_ref[0]) <= TOL_BF16


def test_repeated_calls_are_deterministic():
    x = synthetic.make_replay_inputs([777], 2, 4, 128, 128, dtype="bf16", seed=309)
    O1, S1 = _run(x)
    O2, S2 = _run(x)
    assert torch.equal(S1, S2) and torch.equal(O1, O2)


@pytest.mark.parametrize("with_S0,gate_scale", [(False, 0.1), (True, 0.1), (True, 1e-3)])
def test_scalar_decay_family(with_S0, gate_scale):
    """The scalar-transition (Mamba-2) family on the tensor-core path: no rank-1 projection, so
    the chunk's A and W vanish; ragged tails, an entering state, weak decay."""
    x = synthetic.make_replay_inputs([300, 64, 1, 129], 2, 4, 128, 128, dtype="bf16", seed=311,
                                     with_S0=with_S0, gate_scale=gate_scale)
    O, S = _run(x, scalar_decay=True)
    _check(x, O, S, scalar_decay=True)


# State-only calls with few problems (32-row slices) take the operator-form scan: the chunk's
# d_k x d_k operator K^T Z K is built ahead of the chain and the chain holds one product per chunk.
@pytest.mark.parametrize("with_S0", [False, True])
def test_state_only_ragged_few_problems(with_S0):
    x = synthetic.make_replay_inputs(RAGGED, 2, 4, 128, 128, dtype="bf16", seed=330 + with_S0, unit_qk=False,
                                     with_S0=with_S0)
    _, S = _run(x, state_only=True)
    _check(x, None, S, want_O=False)


def test_state_only_weak_decay_carry():
    x = synthetic.make_replay_inputs([1000, 333], 2, 4, 128, 128, dtype="bf16", seed=332, gate_scale=1e-3,
                                     with_S0=True)
    _, S = _run(x, state_only=True)
    _check(x, None, S, want_O=False)


def test_state_only_three_v_heads_per_key_head():
    x = synthetic.make_replay_inputs([130, 64, 5], 1, 3, 128, 128, dtype="bf16", seed=333, with_S0=True)
    _, S = _run(x, state_only=True)
    _check(x, None, S, want_O=False)


@pytest.mark.parametrize("with_S0", [False, True])
def test_state_only_scalar_decay_family(with_S0):
    x = synthetic.make_replay_inputs([300, 64, 1, 129], 2, 4, 128, 128, dtype="bf16", seed=334, with_S0=with_S0)
    _, S = _run(x, state_only=True, scalar_decay=True)
    _check(x, None, S, want_O=False, scalar_decay=True)


def test_state_only_single_layer_workload():
    x = synthetic.workload_inputs("layer_r3277")
    _, S = _run(x, state_only=True)
    _check(x, None, S, want_O=False)


def test_state_only_matches_outputs_path():
    """The operator-form state equals the state of the call that also writes outputs (another
    grouping of the same products) to the bf16 bar."""
    x = synthetic.make_replay_inputs([700, 90], 2, 4, 128, 128, dtype="bf16", seed=335, with_S0=True)
    _, S1 = _run(x, state_only=True)
    _, S2 = _run(x)
    assert rel_err(host(S1), host(S2)) <= TOL_BF16


def test_state_only_many_problems_64_row_slices():
    """State only with many (tail, head) pairs: the two-product scan on 64-row slices, no outputs."""
    rng = np.random.Generator(np.random.PCG64(336))
    lengths = [int(v) for v in rng.integers(0, 300, size=24)]
    x = synthetic.make_replay_inputs(lengths, 2, 4, 128, 128, dtype="bf16", seed=337, with_S0=True)
    _, S = _run(x, state_only=True)
    _check(x, None, S, want_O=False)
