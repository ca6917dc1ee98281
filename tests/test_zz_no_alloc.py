"""fa_verify_forward_static: the split-KV path for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plugin whose host runtime owns all
device memory and passes it only its inputs and outputs; a serving loop that
reserved nearly all of HBM up front; a loop that cannot take the
synchronisation an allocation may cause). This entry point keeps its
split-KV partials in a library-owned device array instead. The test checks,
through the C ABI, that two calls in a row on different inputs give what the
allocating entry point gives, within the parity tolerances of the suite, and
that a shape whose partials do not fit is refused. The file sorts last so a
run that stops at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import WORKLOADS, with_seed, make_qkv

pytestmark = pytest.mark.gpu

TOL_O_MAX, TOL_O_MEAN, TOL_LSE = 2e-2, 2e-3, 1e-3


def _outputs(w):
    o = torch.full((w.B, w.H, w.Sq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H, w.Sq), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def _allocating(w, q, k, v, n_split):
    o, lse = _outputs(w)
    need = _capi.fa_verify_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d, n_split)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_verify_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal,
                                        w.scale, n_split, ws, need), "fa_verify_forward")
    return o, lse


def _static(w, q, k, v, n_split):
    o, lse = _outputs(w)
    _capi.check(_capi.fa_verify_forward_static(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d,
                                               w.causal, w.scale, n_split),
                "fa_verify_forward_static")
    return o, lse


def _close(a, b):
    (oa, la), (ob, lb) = a, b
    err = (oa.float() - ob.float()).abs()
    assert torch.isfinite(oa.float()).all()
    assert err.max().item() <= TOL_O_MAX and err.mean().item() <= TOL_O_MEAN
    fin = torch.isfinite(lb)
    assert torch.equal(torch.isfinite(la), fin)
    assert (la[fin] - lb[fin]).abs().max().item() <= TOL_LSE


@pytest.mark.parametrize("n_split", [0, 4])
def test_static_scratch_matches_the_allocating_entry_on_two_calls_in_a_row(n_split):
    base = WORKLOADS["verify_b16h32q5k4096d128"]
    inputs = [tuple(t.cuda() for t in make_qkv(with_seed(base, s))) for s in (4, 5)]
    refs = [_allocating(base, *x, n_split) for x in inputs]
    got = [_static(base, *x, n_split) for x in inputs]   # two calls back to back
    torch.cuda.synchronize()
    assert _capi.fa_device_status() == _capi.FA_OK
    for g, r in zip(got, refs):
        _close(g, r)
    # the two inputs really differ, so stale scratch would have shown
    assert not torch.equal(got[0][0], got[1][0])


def test_static_scratch_refuses_partials_beyond_its_size():
    B, H, Sq, Sk, d, n_split = 16, 32, 16, 4096, 128, 8
    assert _capi.fa_verify_workspace_size(B, H, Sq, Sk, d, n_split) > _capi.FA_STATIC_SCRATCH_BYTES
    w = with_seed(WORKLOADS["verify_b16h32q5k4096d128"], 6)
    q = torch.zeros((B, H, Sq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, Sk, d), dtype=torch.bfloat16, device="cuda")
    o, lse = torch.zeros_like(q), torch.zeros((B, H, Sq), dtype=torch.float32, device="cuda")
    st = _capi.fa_verify_forward_static(q, k, k, o, lse, B, H, Sq, Sk, d, 1, w.scale, n_split)
    assert st == _capi.FA_ERR_WORKSPACE
    assert np.all(o.float().cpu().numpy() == 0)
