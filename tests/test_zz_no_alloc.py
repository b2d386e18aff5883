"""The allocation-free draft entry point against the workspace one.

dspark_draft_markov_noalloc serves callers that cannot allocate device
memory (a host framework owning every allocation, or a loop that must not
enter the allocator); it keeps the draft's scratch in a fixed array inside
the library.  Two calls in a row must each reproduce dspark_draft_markov:
the second call checks that the array's leftover contents from the first do
not leak into the result.  This file sorts last so that a run stopping at
the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import workload
from tests._parity import LOGIT_ATOL

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise
    vm = None


def _outputs(B, gamma, dev="cuda"):
    return (torch.empty((B, gamma), dtype=torch.int32, device=dev),
            torch.empty((B, gamma), device=dev), torch.empty((B, gamma), device=dev))


@pytest.mark.parametrize("B,V,r,wdt", [
    (64, 4104, 256, torch.bfloat16),     # tensor-core path, ragged last tile
    (4, 1024, 32, torch.float32),        # CUDA-core path
])
def test_noalloc_matches_workspace_entry_point_twice(B, V, r, wdt):
    w = workload.custom("tiny", B=B, V=V, r=r, w_dtype=wdt, w_std=0.1, seed=B + V)
    inp = workload.inputs(w, device="cuda")
    ws = vm.Workspace(B, w.gamma, V, r)
    ref_tok, ref_lse, ref_z = _outputs(B, w.gamma)
    for call in range(2):
        seed = 17 + call                  # the second call draws different tokens
        vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], ref_tok, ref_lse, ref_z, ws,
                               seed=seed, step=call)
        tok, lse, z = _outputs(B, w.gamma)
        vm.dspark_draft_markov_noalloc(inp["U"], inp["W1"], inp["W2"], inp["anchor"], tok, lse, z,
                                       seed=seed, step=call)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok.cpu().numpy())
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=LOGIT_ATOL, rtol=0)
        np.testing.assert_allclose(z.cpu().numpy(), ref_z.cpu().numpy(), atol=LOGIT_ATOL, rtol=0)


def test_noalloc_at_its_batch_limit_matches_workspace_entry_point():
    """B = 256 is the documented limit at any vocabulary: the b256 vocabulary
    (V = 129280) and the full one (V = 151936) with gamma = 7 must run and
    reproduce dspark_draft_markov."""
    for V, r in ((129280, 128), (151936, 256)):
        w = workload.custom("b256", B=256, V=V, r=r, seed=V)
        inp = workload.inputs(w, device="cuda")
        ws = vm.Workspace(w.B, w.gamma, V, r)
        ref = _outputs(w.B, w.gamma)
        got = _outputs(w.B, w.gamma)
        vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], *ref, ws, seed=3, step=1)
        vm.dspark_draft_markov_noalloc(inp["U"], inp["W1"], inp["W2"], inp["anchor"], *got, seed=3, step=1)
        assert vm.dspark_noalloc_sync_status() == (0, 0)
        np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
        np.testing.assert_allclose(got[1].cpu().numpy(), ref[1].cpu().numpy(), atol=LOGIT_ATOL, rtol=0)
        del inp, ws
        torch.cuda.empty_cache()


def test_noalloc_rejects_sizes_beyond_its_array():
    B, gamma, V, r = 257, 7, 1024, 64
    tok, lse, z = _outputs(B, gamma)
    U = torch.empty((B, gamma, V), device="cuda")
    W1 = torch.empty((V, r), dtype=torch.bfloat16, device="cuda")
    W2 = torch.empty((r, V), dtype=torch.bfloat16, device="cuda")
    anchor = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(vm.DsparkError) as ei:
        vm.dspark_draft_markov_noalloc(U, W1, W2, anchor, tok, lse, z, seed=0)
    assert ei.value.status == -4


def test_noalloc_status_word_reports_range_checks():
    """An anchor outside [0, V) sets the token bit in the fixed array's status
    word; dspark_noalloc_sync_status reports it once and clears it."""
    w = workload.custom("tiny", B=4, V=1024, r=64, w_dtype=torch.bfloat16, seed=9)
    inp = workload.inputs(w, device="cuda")
    inp["anchor"][1] = w.V + 3
    tok, lse, z = _outputs(w.B, w.gamma)
    vm.dspark_draft_markov_noalloc(inp["U"], inp["W1"], inp["W2"], inp["anchor"], tok, lse, z, seed=1)
    st, bits = vm.dspark_noalloc_sync_status()
    assert st == -5 and bits & 1
    assert vm.dspark_noalloc_sync_status() == (0, 0)
