"""spec_tree_verify_stochastic_noalloc: the stochastic verifier for callers
that cannot allocate device memory when they verify (a host framework that
passes the library only its inputs and outputs, or a loop that must not pay
cudaMalloc's device-wide synchronisation).  Its scratch is a fixed device array
inside the library, shared by every call.  Two calls in a row, on different
batches, must each give exactly what the workspace-taking entry point gives
(paths, emitted tokens and statuses are integers: bit-exact)."""
import numpy as np
import pytest
import torch

import workloads as W
import tree_speculative_verification_spec_gb300 as S
from tree_speculative_verification_spec_gb300.pipeline import DeviceBatch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_verification_spec_gb300 import build
    build.build()
    S.lib()


def _outputs(d):
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(path=torch.full((d.B, d.n_max), 7, **i32), accept_len=torch.full((d.B,), 7, **i32),
                emitted=torch.full((d.B, d.n_max), 7, **i32), n_emitted=torch.full((d.B,), 7, **i32),
                status=torch.zeros(d.B, **i32))


def _with_workspace(d):
    o = _outputs(d)
    ws = torch.empty(S.spec_verify_workspace_size(d.B, d.n_max, d.V), dtype=torch.uint8, device="cuda")
    S.spec_tree_verify_stochastic(d.p_logits, d.q_probs, d.tokens, d.parent, d.tree_off, d.uniforms, d.B, d.n_max,
                                  d.V, o["path"], o["accept_len"], o["emitted"], o["n_emitted"], ws, o["status"])
    return o


def _without_workspace(d):
    o = _outputs(d)
    S.spec_tree_verify_stochastic_noalloc(d.p_logits, d.q_probs, d.tokens, d.parent, d.tree_off, d.uniforms, d.B,
                                          d.n_max, d.V, o["path"], o["accept_len"], o["emitted"], o["n_emitted"],
                                          o["status"])
    return o


def test_noalloc_verify_matches_workspace_verify_on_two_calls_in_a_row():
    batches = [DeviceBatch.from_workload(W.config1()),
               DeviceBatch.from_workload(W.small_random(77, B=5, n_range=(1, 50), prefix_range=(0, 1), Hq=2, Hkv=1,
                                                        D=64, V=128256, block_size=16))]
    for d in batches:  # two consecutive calls of the no-allocation entry point
        got = _without_workspace(d)
        ref = _with_workspace(d)
        torch.cuda.synchronize()
        for k in ("path", "accept_len", "emitted", "n_emitted", "status"):
            assert torch.equal(got[k], ref[k]), k
        assert int(ref["accept_len"].min()) >= 1


def test_noalloc_verify_rejects_batches_beyond_its_scratch():
    L = S.lib()
    assert L.spec_tree_verify_stochastic_noalloc(*[None] * 6, 1 << 15, 8, 100, *[None] * 6) == S.SPEC_ERR_UNSUPPORTED
    assert L.spec_tree_verify_stochastic_noalloc(*[None] * 6, 1024, 1024, 100, *[None] * 6) == S.SPEC_ERR_UNSUPPORTED
