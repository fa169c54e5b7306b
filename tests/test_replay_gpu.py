"""GPU parity of gdn_replay / gdn_chunk_operator / gdn_compose against the fp64 oracle.

Every call goes through the C ABI (libgdn.so via the thin binding); the
oracle runs on the host on the same seeded inputs.  Errors are relative
Frobenius norms over whole tensors.  Tolerances: 1e-5 for fp32 inputs,
3e-3 for bf16 inputs (fp32 accumulation and state; O is rounded to bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_state_chunked_gb300 import _lib, api, synthetic
from tests.gpu_util import TOL_BF16, TOL_F32, host, oracle_replay, rel_err, to_device

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


def test_tiny_config_fp32():
    """1 sequence, 2 heads, d_k = d_v = 64, 256-token tail, fp32, zero initial state."""
    x = synthetic.workload_inputs("tiny")
    O, S = _run(x)
    S_ref, O_ref = oracle_replay(x)
    assert rel_err(host(S), S_ref) <= TOL_F32
    assert rel_err(host(O), O_ref) <= TOL_F32


RAGGED = [1, 63, 64, 65, 130, 0, 200]


@pytest.mark.parametrize("d_k,d_v", [(64, 32), (128, 128), (16, 64), (128, 8)])
@pytest.mark.parametrize("with_S0", [False, True])
def test_ragged_batch_fp32(d_k, d_v, with_S0):
    x = synthetic.make_replay_inputs(RAGGED, 2, 4, d_k, d_v, dtype="f32", seed=100 + d_k + d_v,
                                     unit_qk=False, with_S0=with_S0)
    O, S = _run(x, scale=0.5)
    S_ref, O_ref = oracle_replay(x, scale=0.5)
    assert rel_err(host(S), S_ref) <= TOL_F32
    assert rel_err(host(O), O_ref) <= TOL_F32


def test_without_l2norm_fp32():
    x = synthetic.make_replay_inputs([77, 129], 1, 2, 32, 32, dtype="f32", seed=7, with_S0=True)
    O, S = _run(x, l2norm_qk=False)
    S_ref, O_ref = oracle_replay(x, l2norm_qk=False)
    assert rel_err(host(S), S_ref) <= TOL_F32
    assert rel_err(host(O), O_ref) <= TOL_F32


def test_state_only_leaves_outputs_alone():
    x = synthetic.make_replay_inputs([90, 3], 2, 2, 64, 64, dtype="f32", seed=8)
    d = to_device(x)
    _, S = api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], state_only=True)
    torch.cuda.synchronize()
    S_ref, _ = oracle_replay(x, want_O=False)
    assert rel_err(host(S), S_ref) <= TOL_F32


def test_rows_outside_sequences_are_not_written():
    x = synthetic.make_replay_inputs([50, 40], 1, 2, 32, 32, dtype="f32", seed=9)
    d = to_device(x)
    cu = torch.tensor([0, 50, 80], dtype=torch.int32, device="cuda")  # last 10 tokens belong to no sequence
    O = torch.full((90, 2, 32), 7.0, device="cuda")
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, O_out=O)
    torch.cuda.synchronize()
    assert torch.all(O[80:] == 7.0)
    S_ref, O_ref = oracle.replay(x.q, x.k, x.v, x.g, x.beta, [0, 50, 80])
    assert rel_err(host(O[:80]), O_ref[:80]) <= TOL_F32


def test_in_place_state_update():
    x = synthetic.make_replay_inputs([70, 20], 1, 2, 32, 32, dtype="f32", seed=10, with_S0=True)
    d = to_device(x)
    S = d["S0"].clone()
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S, S_out=S, state_only=True)
    torch.cuda.synchronize()
    S_ref, _ = oracle_replay(x, want_O=False)
    assert rel_err(host(S), S_ref) <= TOL_F32


def test_malformed_cu_seqlens_sets_status_and_skips_sequence():
    x = synthetic.make_replay_inputs([30, 30, 30], 1, 1, 16, 16, dtype="f32", seed=11)
    d = to_device(x)
    cu = torch.tensor([0, 30, 20, 90], dtype=torch.int32, device="cuda")  # sequence 1 runs backwards
    S = torch.full((3, 1, 16, 16), 5.0, device="cuda")
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S_out=S, state_only=True)
    with pytest.raises(_lib.GdnError) as ei:
        api.gdn_get_status()
    assert ei.value.code == _lib.GDN_ERR_SHAPE
    api.gdn_get_status()  # the status is cleared once read
    assert torch.all(S[1] == 5.0)
    S_ref, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, [0, 30], want_O=False)
    assert rel_err(host(S[0]), S_ref[0]) <= TOL_F32


def test_overlapping_forward_ranges_are_skipped():
    """[0, T, 0, T]: the ranges after the step back are skipped and reported (fp32 path)."""
    T = 100
    x = synthetic.make_replay_inputs([T], 1, 2, 32, 32, dtype="f32", seed=12)
    d = to_device(x)
    cu = torch.tensor([0, T, 0, T], dtype=torch.int32, device="cuda")
    S = torch.full((3, 2, 32, 32), 5.0, device="cuda")
    api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S_out=S, state_only=True)
    with pytest.raises(_lib.GdnError) as ei:
        api.gdn_get_status()
    assert ei.value.code == _lib.GDN_ERR_SHAPE
    assert torch.all(S[1] == 5.0) and torch.all(S[2] == 5.0)
    S_ref, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, [0, T], want_O=False)
    assert rel_err(host(S[0]), S_ref[0]) <= TOL_F32


def test_precise_path_on_bf16_inputs():
    x = synthetic.make_replay_inputs(RAGGED, 2, 4, 128, 128, dtype="bf16", seed=12, with_S0=True)
    O, S = _run(x, precise=True)
    S_ref, O_ref = oracle_replay(x)
    assert rel_err(host(S), S_ref) <= TOL_F32
    assert rel_err(host(O), O_ref) <= TOL_BF16


# ------------------------------------------------------------------ chunk operator and composition

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_operator_matches_oracle(dtype):
    x = synthetic.make_replay_inputs([200, 1, 64, 129], 2, 4, 64, 32, dtype=dtype, seed=13, gate_scale=1e-3)
    d = to_device(x)
    T, Sl = api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu_seqlens"])
    torch.cuda.synchronize()
    T_ref, Sl_ref = oracle.chunk_operator(x.k, x.g, x.beta, x.v, x.cu_seqlens)
    assert rel_err(host(T), T_ref) <= TOL_F32
    assert rel_err(host(Sl), Sl_ref) <= TOL_F32


def _ops_on_device(T, layout):
    """The K operators as a list of device tensors.  "one_array": views of one [K, ...] tensor
    (one stride between operators: the tensor-map kernel); "scattered": views of one tensor at
    permuted positions (no common stride: the kernel that copies rows one by one)."""
    K = T.shape[0]
    if layout == "one_array":
        Td = torch.from_numpy(np.ascontiguousarray(T)).cuda()
        return [Td[j] for j in range(K)]
    # reversed slots, the first one step further out: a negative stride for K = 2, none for K > 2
    perm = [K - 1 - j + (1 if j == 0 else 0) for j in range(K)]
    big = torch.zeros((K + 2,) + T.shape[1:], dtype=torch.float32, device="cuda")
    for j in range(K):
        big[perm[j]] = torch.from_numpy(T[j]).cuda()
    return [big[perm[j]] for j in range(K)]


@pytest.mark.parametrize("layout", ["one_array", "scattered"])
def test_compose_matches_oracle_closed_form(layout):
    rng = np.random.Generator(np.random.PCG64(14))
    K, h, dk, dv = 6, 4, 128, 128
    T = (rng.standard_normal((K, h, dk, dk)) / np.sqrt(dk)).astype(np.float32)
    Sl = rng.standard_normal((K, h, dv, dk)).astype(np.float32)
    S_in = rng.standard_normal((h, dv, dk)).astype(np.float32)
    Td = _ops_on_device(T, layout)
    Sd = [torch.from_numpy(Sl[j]).cuda() for j in range(K)]
    out = api.gdn_compose(Td, Sd, torch.from_numpy(S_in).cuda())
    out0 = api.gdn_compose(Td, Sd, None)
    torch.cuda.synchronize()
    assert rel_err(host(out), oracle.compose(T, Sl, S_in)) <= TOL_F32
    assert rel_err(host(out0), oracle.compose(T, Sl, None)) <= TOL_F32


@pytest.mark.parametrize("layout", ["one_array", "scattered"])
@pytest.mark.parametrize("K", [0, 1, 2, 3])
def test_compose_edge_counts(K, layout):
    """K = 0 copies S_in (or writes zeros); K = 1, 2 and 3 exercise the first and last steps of
    the tensor-core composition (128-dim heads) and both copy buffers on their own."""
    rng = np.random.Generator(np.random.PCG64(40 + K))
    h, d = 3, 128
    T = (rng.standard_normal((K, h, d, d)) / np.sqrt(d)).astype(np.float32)
    Sl = rng.standard_normal((K, h, d, d)).astype(np.float32)
    S_in = rng.standard_normal((h, d, d)).astype(np.float32)
    Td = _ops_on_device(T, layout) if K else []
    Sd = [torch.from_numpy(Sl[j]).cuda() for j in range(K)]
    out = api.gdn_compose(Td, Sd, torch.from_numpy(S_in).cuda())
    torch.cuda.synchronize()
    assert rel_err(host(out), oracle.compose(T, Sl, S_in)) <= TOL_F32
    if K == 0:  # nothing to compose and no entering state: the binding refuses
        with pytest.raises(ValueError):
            api.gdn_compose(Td, Sd, None)
    else:
        out0 = api.gdn_compose(Td, Sd, None)
        torch.cuda.synchronize()
        assert rel_err(host(out0), oracle.compose(T, Sl, None)) <= TOL_F32


@pytest.mark.parametrize("layout", ["one_array", "scattered"])
def test_compose_long_chain(layout):
    """K = 40: every copy buffer and barrier phase of the tensor-core composition wraps many
    times; the error stays within the fp32 tolerance over the whole chain."""
    rng = np.random.Generator(np.random.PCG64(77))
    K, h, d = 40, 2, 128
    T = (rng.standard_normal((K, h, d, d)) / np.sqrt(d)).astype(np.float32)
    Sl = rng.standard_normal((K, h, d, d)).astype(np.float32)
    S_in = rng.standard_normal((h, d, d)).astype(np.float32)
    Td = _ops_on_device(T, layout)
    Sd = [torch.from_numpy(Sl[j]).cuda() for j in range(K)]
    out = api.gdn_compose(Td, Sd, torch.from_numpy(S_in).cuda())
    torch.cuda.synchronize()
    api.gdn_get_status()
    assert rel_err(host(out), oracle.compose(T, Sl, S_in)) <= TOL_F32


def test_composed_chunks_equal_sequential_replay():
    """LinearKV composition passage: composing isolated-chunk operators is exact, so
    compose(chunk operators) on the GPU equals the GPU's own sequential replay."""
    pieces = [300, 64, 1, 250]
    x = synthetic.make_replay_inputs([sum(pieces)], 2, 4, 64, 64, dtype="f32", seed=15, gate_scale=1e-3)
    d = to_device(x)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(pieces)]), dtype=torch.int32, device="cuda")
    T, Sl = api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], cu)
    SK = api.gdn_compose([T[j] for j in range(len(pieces))], [Sl[j] for j in range(len(pieces))])
    _, S = api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], state_only=True)
    torch.cuda.synchronize()
    S_ref, _ = oracle_replay(x, want_O=False)
    assert rel_err(host(SK), S_ref[0]) <= TOL_F32
    assert rel_err(host(S[0]), S_ref[0]) <= TOL_F32


@pytest.mark.parametrize("layout", ["one_array", "scattered"])
@pytest.mark.parametrize("K", [1, 5])
def test_compose_wait_that_runs_out_reports_timeout_then_recovers(K, layout):
    """The bounded-wait path without a fault: with a wait limit of zero the first wait on the
    MMAs gives up, the kernel lets its issued MMAs finish and reports GDN_ERR_TIMEOUT; the
    context stays usable and the next call (default limit) is correct."""
    rng = np.random.Generator(np.random.PCG64(60 + K))
    h, d = 4, 128
    T = (rng.standard_normal((K, h, d, d)) / np.sqrt(d)).astype(np.float32)
    Sl = rng.standard_normal((K, h, d, d)).astype(np.float32)
    Td = _ops_on_device(T, layout)
    Sd = [torch.from_numpy(Sl[j]).cuda() for j in range(K)]
    api.gdn_set_wait_limit_ns(0)
    api.gdn_compose(Td, Sd, None)
    with pytest.raises(_lib.GdnError) as ei:
        api.gdn_get_status()
    assert ei.value.code == _lib.GDN_ERR_TIMEOUT
    out = api.gdn_compose(Td, Sd, None)  # the hook was cleared: default bound
    torch.cuda.synchronize()
    api.gdn_get_status()
    assert rel_err(host(out), oracle.compose(T, Sl, None)) <= TOL_F32


@pytest.mark.parametrize("scalar", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_operator_128_dim_heads(dtype, scalar):
    """128-dim heads: the augmented-state scan on tcgen05 in split tf32 (fp32 and bf16 inputs),
    ragged sequences (1, 64, 129, 200 tokens), weak gates so that T_C is far from zero."""
    x = synthetic.make_replay_inputs([200, 1, 64, 129, 3], 2, 4, 128, 128, dtype=dtype, seed=31 + int(scalar),
                                     gate_scale=1e-3)
    d = to_device(x)
    T, Sl = api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu_seqlens"], scalar_decay=scalar)
    torch.cuda.synchronize()
    api.gdn_get_status()
    T_ref, Sl_ref = oracle.chunk_operator(x.k, x.g, x.beta, x.v, x.cu_seqlens, scalar_decay=scalar)
    assert rel_err(host(T), T_ref) <= TOL_F32
    assert rel_err(host(Sl), Sl_ref) <= TOL_F32
    for j in range(x.n_seqs):  # every chunk on its own (the 1- and 3-token ones included)
        assert rel_err(host(T[j]), T_ref[j]) <= TOL_F32
        assert rel_err(host(Sl[j]), Sl_ref[j]) <= TOL_F32


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_state_only_fp32_accurate_128_dim_heads(dtype):
    """State-only replay on the fp32-accurate path with 128-dim heads (fp32 inputs, or bf16 with
    GDN_PRECISE) and an entering state: the same tensor-core scan without the transition rows."""
    x = synthetic.make_replay_inputs([333, 64, 1, 130], 2, 4, 128, 128, dtype=dtype, seed=33, with_S0=True,
                                     gate_scale=1e-3)
    O, S = _run(x, state_only=True, precise=(dtype == "bf16"))
    S_ref, _ = oracle_replay(x, want_O=False)
    assert rel_err(host(S), S_ref) <= TOL_F32


def test_scalar_decay_family_fp32_and_chunk_operator():
    """The scalar-transition (Mamba-2) family on the fp32 path, and its chunk operator: T_C is
    (prod alpha) I and S_local matches the oracle."""
    x = synthetic.make_replay_inputs([200, 1, 64, 129], 2, 4, 64, 32, dtype="f32", seed=15, with_S0=True,
                                     gate_scale=1e-2)
    O, S = _run(x, scalar_decay=True)
    S_ref, O_ref = oracle_replay(x, scalar_decay=True)
    assert rel_err(host(S), S_ref) <= TOL_F32
    assert rel_err(host(O), O_ref) <= TOL_F32
    d = to_device(x)
    T, Sl = api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu_seqlens"], scalar_decay=True)
    torch.cuda.synchronize()
    api.gdn_get_status()
    T_ref, Sl_ref = oracle.chunk_operator(x.k, x.g, x.beta, x.v, x.cu_seqlens, scalar_decay=True)
    assert rel_err(host(T), T_ref) <= TOL_F32
    assert rel_err(host(Sl), Sl_ref) <= TOL_F32
