"""gdn_replay_noalloc, the entry point for callers that cannot allocate device memory.

Some callers of this library cannot allocate GPU memory at call time (for
example a serving process that reserves nearly all HBM for its cache when it
starts and forbids allocations afterwards).  gdn_replay_noalloc serves them by
taking its scratch from a fixed static device array instead of a pool.  This
test calls it through the C ABI twice in a row, on different inputs (so a stale
array from the first call would show in the second), and checks each result
against gdn_replay's and against the fp64 oracle's at the tolerance of the
other bf16 parity tests.  It also
checks that a problem larger than the static array is refused up front.  The
file is named so that pytest collects it last.
"""
import pytest
import torch

from gated_deltanet_state_chunked_gb300 import _lib, api, synthetic
from tests.gpu_util import TOL_BF16, TOL_F32, host, oracle_replay, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    _lib.load(build=True)
    torch.cuda.init()


def _both(x):
    d = to_device(x)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["S0"])
    O_ref, S_ref = api.gdn_replay(*args)
    O = torch.empty_like(O_ref)
    S = torch.empty_like(S_ref)
    api.gdn_replay_noalloc(*args, O, S)
    torch.cuda.synchronize()
    api.gdn_get_status()
    return (O, S), (O_ref, S_ref)


def test_matches_gdn_replay_on_two_calls_in_a_row():
    """Each call's result agrees with gdn_replay's and with the fp64 oracle's."""
    first = synthetic.make_replay_inputs([700, 333, 64], 2, 4, 128, 128, dtype="bf16", seed=501, with_S0=True)
    second = synthetic.make_replay_inputs([1300, 5], 2, 4, 128, 128, dtype="bf16", seed=502, unit_qk=False)
    for x in (first, second):
        (O, S), (O_ref, S_ref) = _both(x)
        assert rel_err(host(S), host(S_ref)) <= TOL_BF16
        assert rel_err(host(O), host(O_ref)) <= TOL_BF16
        S_or, O_or = oracle_replay(x)
        assert rel_err(host(S), S_or) <= TOL_BF16
        assert rel_err(host(O), O_or) <= TOL_BF16


@pytest.mark.parametrize("d_k,d_v", [(128, 128), (64, 32)])
def test_fp32_inputs_one_pass_path_matches_the_oracle(d_k, d_v):
    """fp32 inputs need no scratch here: the fp32 path computes the chunk-shared quantities in
    every row slice (one pass) instead of reading records.  Checked against the fp64 oracle."""
    x = synthetic.make_replay_inputs([300, 77, 1], 2, 4, d_k, d_v, dtype="f32", seed=504, with_S0=True)
    d = to_device(x)
    O = torch.empty((x.total_tokens, 4, d_v), dtype=torch.float32, device="cuda")
    S = torch.empty((3, 4, d_v, d_k), dtype=torch.float32, device="cuda")
    api.gdn_replay_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["S0"], O, S)
    torch.cuda.synchronize()
    api.gdn_get_status()
    S_ref, O_ref = oracle_replay(x)
    assert rel_err(host(S), S_ref) <= TOL_F32
    assert rel_err(host(O), O_ref) <= TOL_F32


def test_single_layer_3277_token_tail_fits():
    x = synthetic.workload_inputs("layer_r3277")
    (O, S), (O_ref, S_ref) = _both(x)
    assert rel_err(host(S), host(S_ref)) <= TOL_BF16
    assert rel_err(host(O), host(O_ref)) <= TOL_BF16
    S_or, O_or = oracle_replay(x)
    assert rel_err(host(S), S_or) <= TOL_BF16
    assert rel_err(host(O), O_or) <= TOL_BF16


def test_rejects_a_problem_beyond_the_static_scratch():
    x = synthetic.make_replay_inputs([8192], 16, 32, 128, 128, dtype="bf16", seed=503)
    d = to_device(x)
    O = torch.empty((x.total_tokens, 32, 128), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((1, 32, 128, 128), device="cuda")
    with pytest.raises(_lib.GdnError) as ei:
        api.gdn_replay_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None, O, S)
    assert ei.value.code == _lib.GDN_ERR_NOMEM
