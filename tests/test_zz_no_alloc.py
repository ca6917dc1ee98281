"""fa_verify_forward_static: the split-KV path for callers that cannot allocate.

Some callers cannot call cudaMalloc: a plugin whose host runtime owns all
device memory and passes it only its inputs and outputs; a serving loop that
reserved nearly all of HBM up front, where a late allocation can fail; a loop
that cannot take the synchronisation an allocation may cause. This entry point
keeps its split-KV partials in a library-owned device array instead.

Both entry points run the same kernels with the same split count on the same
inputs, so the static one must agree with the allocating one bit for bit; a
stale-scratch or offset bug would break that equality. The checks, through the
C ABI: two calls in a row on different inputs, each equal to the allocating
entry point and to the fp64 oracle within the suite's bars; the automatic
split count lowered to fit the array at Sq = 16 (where the automatic count of
the allocating entry would not fit); and an explicit split count that does not
fit refused. The file sorts last so a run that stops at the first failure has
run every other test first.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import WORKLOADS, custom, make_qkv, sample_rows, with_seed
from parity import compare, gather_rows

pytestmark = pytest.mark.gpu


def _outputs(B, H, Sq, d):
    o = torch.full((B, H, Sq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def _allocating(w, q, k, v, n_split):
    o, lse = _outputs(w.B, w.H, w.Sq, w.d)
    need = _capi.fa_verify_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d, n_split)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_verify_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal,
                                        w.scale, n_split, ws, need), "fa_verify_forward")
    torch.cuda.synchronize()
    return o, lse


def _static(w, q, k, v, n_split):
    o, lse = _outputs(w.B, w.H, w.Sq, w.d)
    _capi.check(_capi.fa_verify_forward_static(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d,
                                               w.causal, w.scale, n_split),
                "fa_verify_forward_static")
    return o, lse


def _equal(a, b):
    (oa, la), (ob, lb) = a, b
    assert torch.isfinite(oa.float()).all()
    assert torch.equal(oa, ob), (oa.float() - ob.float()).abs().max().item()
    assert torch.equal(la, lb)


def _against_oracle(w, inputs_cpu, got, n_rows=64):
    rows = sample_rows(w, n_total=n_rows)
    o_ref, l_ref = oracle.attention(*inputs_cpu, w.causal, w.scale, rows=rows)
    og, lg = gather_rows(got[0].float().cpu(), got[1].cpu(), rows)
    compare(og, lg, o_ref, l_ref)


def _static_splits(w):
    """The count the static entry uses for n_split = 0: the automatic count,
    lowered to the largest one whose partials fit the library's array."""
    ns = _capi.fa_verify_auto_splits(w.B, w.H, w.Sq, w.Sk, w.d)
    while ns > 1 and _capi.fa_verify_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d, ns) > \
            _capi.FA_STATIC_SCRATCH_BYTES:
        ns -= 1
    return ns


@pytest.mark.parametrize("n_split", [0, 4])
def test_static_scratch_matches_the_allocating_entry_on_two_calls_in_a_row(n_split):
    base = WORKLOADS["verify_b16h32q5k4096d128"]
    cpu = [make_qkv(with_seed(base, s)) for s in (4, 5)]
    inputs = [tuple(t.cuda() for t in x) for x in cpu]
    ns = n_split or _static_splits(base)
    refs = [_allocating(base, *x, ns) for x in inputs]
    got = [_static(base, *x, n_split) for x in inputs]   # two calls back to back
    torch.cuda.synchronize()
    assert _capi.fa_device_status() == _capi.FA_OK
    for g, r in zip(got, refs):
        _equal(g, r)
    for x, g in zip(cpu, got):
        _against_oracle(base, x, g)


def test_automatic_split_count_is_lowered_to_fit_the_array():
    """Sq = 16: the allocating entry's automatic count needs more partials than
    the array holds; the static entry lowers it and still runs."""
    w = custom(16, 32, 16, 4096, 128, True, seed=9)
    auto = _capi.fa_verify_auto_splits(w.B, w.H, w.Sq, w.Sk, w.d)
    assert auto > 1
    assert _capi.fa_verify_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d, auto) > \
        _capi.FA_STATIC_SCRATCH_BYTES
    ns = _static_splits(w)
    cpu = make_qkv(w)
    q, k, v = (t.cuda() for t in cpu)
    got = _static(w, q, k, v, 0)
    ref = _allocating(w, q, k, v, ns)
    torch.cuda.synchronize()
    assert _capi.fa_device_status() == _capi.FA_OK
    _equal(got, ref)
    _against_oracle(w, cpu, got)


def test_static_scratch_refuses_an_explicit_split_beyond_its_size():
    B, H, Sq, Sk, d, n_split = 16, 32, 16, 4096, 128, 8
    assert _capi.fa_verify_workspace_size(B, H, Sq, Sk, d, n_split) > _capi.FA_STATIC_SCRATCH_BYTES
    w = with_seed(WORKLOADS["verify_b16h32q5k4096d128"], 6)
    q = torch.zeros((B, H, Sq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, Sk, d), dtype=torch.bfloat16, device="cuda")
    o, lse = torch.zeros_like(q), torch.zeros((B, H, Sq), dtype=torch.float32, device="cuda")
    st = _capi.fa_verify_forward_static(q, k, k, o, lse, B, H, Sq, Sk, d, 1, w.scale, n_split)
    assert st == _capi.FA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert np.all(o.float().cpu().numpy() == 0)
