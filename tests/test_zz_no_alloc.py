"""spec_tree_attention_noalloc: tree attention for callers that cannot
allocate device memory where they run it (a host framework that passes the
library only the tensors it owns, or a serving loop whose graphs are captured
once and must not pay cudaMalloc's device-wide synchronisation).  When the plan
splits a long key range over several CTAs, the partial outputs of the splits
go to a fixed scratch array inside the library, shared by every call.

Two calls in a row, on different shapes whose plans split their keys (so the
scratch really holds partials, and the second call starts from the first
call's leftovers), must each match the CPU oracle and spec_tree_attention with
a caller-allocated workspace, within the attention tolerance of the other
tests.  That the plan these calls take needs scratch is shown by the
workspace entry point refusing to run without a workspace.  This file is
collected last and passes alone or after the rest of the suite."""
import numpy as np
import pytest
import torch

import workloads as W
import tree_speculative_verification_spec_gb300 as S
from tree_speculative_verification_spec_gb300.pipeline import DeviceBatch, VerifyPass
from parity import attn_tolerance_ok, bf16_bits_to_f32, oracle_attention

pytestmark = pytest.mark.gpu

CASES = [dict(seed=91, B=1, n_range=(16, 16), prefix_range=(12000, 12000), Hq=32, Hkv=8, D=128, block_size=64),
         dict(seed=92, B=2, n_range=(5, 24), prefix_range=(5000, 9000), Hq=16, Hkv=2, D=64, block_size=16)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_verification_spec_gb300 import build
    build.build()
    S.lib()


def _args(d, mask):
    return (d.q, d.k_cache, d.v_cache, d.block_table, d.max_blocks, d.block_size, d.num_blocks, d.prefix_len,
            d.tree_off, mask, d.B, d.T, d.n_max, d.max_prefix, d.Hq, d.Hkv, d.D, d.scale)


def test_noalloc_attention_matches_workspace_attention_on_two_calls_in_a_row():
    for c in CASES:
        c = dict(c)
        w = W.small_random(c.pop("seed"), V=16, dtype=W.BF16, **c)
        d = DeviceBatch.from_workload(w)
        vp = VerifyPass(d)
        vp.mask_build()
        ws_bytes = S.spec_attention_workspace_size(d.B, d.T, d.n_max, d.max_prefix, d.Hq, d.Hkv, d.D)
        assert 256 < ws_bytes <= S.SPEC_ATTN_NOALLOC_BYTES  # the plan splits the keys; the scratch holds them
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out_ref, st_ref = torch.full_like(d.q, 7.0), torch.zeros(d.B, dtype=torch.int32, device="cuda")
        out_na, st_na = torch.full_like(d.q, -7.0), torch.zeros(d.B, dtype=torch.int32, device="cuda")
        # the plan of this call (AUTO, bf16) needs scratch: without a workspace it is refused
        with pytest.raises(S.SpecError) as e:
            S.spec_tree_attention(*_args(d, vp.mask), out_ref, None, st_ref)
        assert e.value.code == S.SPEC_ERR_WORKSPACE
        S.spec_tree_attention(*_args(d, vp.mask), out_ref, ws, st_ref)
        S.spec_tree_attention_noalloc(*_args(d, vp.mask), out_na, st_na)
        torch.cuda.synchronize()
        assert st_ref.cpu().tolist() == st_na.cpu().tolist() == [0] * d.B
        ref = out_ref.float().cpu().numpy()
        got = out_na.float().cpu().numpy()
        assert np.isfinite(ref).all()
        assert attn_tolerance_ok(got, ref, w.dtype).all(), float(np.abs(got - ref).max())
        # and directly against the oracle (fp64 attention rounded to bf16)
        ora, _, s_ora = oracle_attention(w)
        assert (s_ora == 0).all()
        ora32 = bf16_bits_to_f32(ora).reshape(got.shape)
        assert attn_tolerance_ok(got, ora32, w.dtype).all(), float(np.abs(got - ora32).max())


def test_noalloc_attention_rejects_shapes_beyond_its_scratch():
    """A plan whose partials exceed the scratch array returns
    SPEC_ERR_UNSUPPORTED before touching any pointer or launching."""
    L = S.lib()
    need = S.spec_attention_workspace_size(1, 1024, 1024, 60000, 64, 8, 128)
    assert need > S.SPEC_ATTN_NOALLOC_BYTES
    rc = L.spec_tree_attention_noalloc(None, None, None, None, 1, 64, 1, None, None, None, 1, 1024, 1024, 60000, 64, 8,
                                       128, S.SPEC_BF16, 0.088, None, None, S.SPEC_ATTN_AUTO, None)
    assert rc == S.SPEC_ERR_UNSUPPORTED
