"""GPU parity: the sm_103a kernels, called through the C ABI, against the fp64
oracle on the same seeded bf16 inputs, element by element.

Sizes are chosen so the oracle finishes in seconds while the kernels still run
several query/key tiles and a ragged tail; the full-size workloads are checked
on sampled rows in the same launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_03_gb300 import _capi
from exact_tiled_attention_03_gb300.inputs import WORKLOADS, custom, make_qkv, sample_rows, with_seed
from parity import compare, gather_rows, oracle_full, oracle_rows, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _capi.load()


# ---------------------------------------------------------------- building blocks
@pytest.mark.parametrize("n", [64, 128])
@pytest.mark.parametrize("k", [64, 128])
@pytest.mark.parametrize("b_mn_major", [0, 1])
def test_tcgen05_descriptors_one_tile_gemm(n, k, b_mn_major):
    """One TMA -> SMEM -> tcgen05.mma -> TMEM tile, against a CPU matmul."""
    g = torch.Generator().manual_seed(n * 7 + k + b_mn_major)
    a = torch.randn(128, k, generator=g).to(torch.bfloat16)
    b = torch.randn(n, k, generator=g).to(torch.bfloat16)          # B as N x K
    b_dev = (b.t().contiguous() if b_mn_major else b).cuda()        # K x N when MN-major
    c = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    _capi.check(_capi.fa_selftest_umma(a.cuda(), b_dev, c, n, k, b_mn_major), "selftest_umma")
    torch.cuda.synchronize()
    ref = a.double() @ b.double().t()
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3 * math.sqrt(k), err


@pytest.mark.parametrize("n", [64, 128])
@pytest.mark.parametrize("k", [64, 128])
@pytest.mark.parametrize("b_mn_major", [0, 1])
def test_tcgen05_a_operand_from_tensor_memory(n, k, b_mn_major):
    """A written to TMEM (two bf16 per column, even element low) and read by the MMA."""
    g = torch.Generator().manual_seed(n * 11 + k + b_mn_major)
    a = torch.randn(128, k, generator=g).to(torch.bfloat16)
    b = torch.randn(n, k, generator=g).to(torch.bfloat16)
    b_dev = (b.t().contiguous() if b_mn_major else b).cuda()
    c = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    _capi.check(_capi.fa_selftest_umma_ts(a.cuda(), b_dev, c, n, k, b_mn_major), "selftest_umma_ts")
    torch.cuda.synchronize()
    ref = a.double() @ b.double().t()
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3 * math.sqrt(k), err


def test_mufu_microbenchmark_runs():
    """The exp2 throughput kernel the benchmark uses for the softmax's second bound."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.full((sms * 256,), float("nan"), dtype=torch.float32, device="cuda")
    _capi.check(_capi.fa_selftest_mufu(out, sms, 64), "mufu")
    torch.cuda.synchronize()
    v = out.cpu()
    assert torch.isfinite(v).all()
    # each chain settles at the fixed point of x = -0.5 * 2^x - 0.25 (about -0.59)
    assert ((v / 8 + 0.59).abs() < 0.02).all()


def test_elect_sync_picks_the_same_lane_every_time():
    """The warp-wide MMA issue loops let elect.sync pick the issuing lane for
    each MMA and each commit separately; a commit tracks only its own thread's
    MMAs, so every election of a converged warp must pick the same lane."""
    trials = 256
    lanes = torch.full((4 * trials,), -1, dtype=torch.int32, device="cuda")
    _capi.check(_capi.fa_selftest_elect(lanes, trials), "elect")
    torch.cuda.synchronize()
    assert (lanes.cpu() == 0).all()


def test_mma_rate_of_the_operand_forms():
    """The gradient kernels issue only 128-wide MMAs because two 64-wide halves
    take longer than one 128-wide MMA of the same work (measured 45-54 against 64
    cycles per K = 16 instruction). Cycle counts do not depend on the clock."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.empty(sms, dtype=torch.int64, device="cuda")
    per = {}
    for mode in range(7):
        for _ in range(2):  # the first launch of a form warms the tensor pipe up
            _capi.check(_capi.fa_selftest_mma_rate(cyc, mode, sms, 1000), "mma_rate")
        torch.cuda.synchronize()
        c = cyc.cpu()
        assert (c > 0).all()
        per[mode] = c.double().median().item() / (1000 * (2 if mode == 4 else 1))
    assert _capi.fa_device_status() == _capi.FA_OK
    for mode in (0, 2, 4):          # full-width forms run near the nominal 512
        assert 480 < per[mode] < 620, per
    for half, full in ((1, 0), (3, 2)):
        assert per[half] > 1.25 * per[full], per
    for mode in (5, 6):             # an E4M3 product is faster than a bf16 one
        assert 100 < per[mode] < per[0], per
    assert _capi.fa_selftest_mma_rate(cyc, 7, 1, 1) == _capi.FA_ERR_UNSUPPORTED
    assert _capi.fa_selftest_mma_rate(None, 0, 1, 1) == _capi.FA_ERR_INVALID_ARG


def test_bounded_wait_reports_a_timeout_without_faulting():
    """A wait on a barrier nothing completes gives up, sets the status word, returns."""
    assert _capi.fa_device_status() == _capi.FA_OK
    _capi.check(_capi.fa_selftest_wait_timeout(50_000_000), "selftest_wait")
    assert _capi.fa_device_status() == _capi.FA_ERR_TIMEOUT
    assert _capi.fa_device_status() == _capi.FA_OK  # read-and-clear


# ---------------------------------------------------------------- tiny workload, every path
@pytest.mark.parametrize("name", ["tiny_b1h1s256d64_noncausal", "tiny_b1h1s256d64_causal"])
@pytest.mark.parametrize("entry", ["fa_forward", "fa_prefill_forward", "fa_reference_forward_simt"])
def test_tiny_workload(name, entry):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w)
    o, lse = run(entry, q, k, v, w.causal, w.scale)
    ro, rl = oracle_full(q, k, v, w.causal, w.scale)
    compare(o, lse, ro, rl)


# ---------------------------------------------------------------- prefill kernel edge cases
PREFILL_CASES = [
    # B, H, Sq, Sk, d, causal
    (1, 2, 17, 17, 64, True),
    (1, 2, 127, 127, 128, True),
    (1, 1, 128, 128, 128, True),
    (1, 1, 129, 129, 128, True),
    (1, 2, 255, 255, 64, True),
    (1, 1, 256, 256, 128, True),
    (1, 1, 257, 257, 128, True),
    (2, 1, 1000, 1000, 128, True),
    (1, 1, 1000, 1000, 64, False),
    (1, 3, 129, 300, 128, False),
    (1, 2, 300, 129, 64, False),
    (1, 1, 200, 1000, 128, True),   # bottom-right: Sq < Sk
    (1, 1, 300, 100, 128, True),    # Sq > Sk: the first 200 rows see nothing
    (1, 1, 513, 700, 64, True),
    (1, 1, 17, 1, 128, True),
    (1, 1, 33, 1, 64, False),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
def test_prefill_edge_shapes(case):
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq * 31 + Sk)
    q, k, v = make_qkv(w)
    o, lse = run("fa_prefill_forward", q, k, v, causal, w.scale)
    ro, rl = oracle_full(q, k, v, causal, w.scale)
    compare(o, lse, ro, rl)


def test_prefill_large_logits_rescale():
    """Q x 8: logits of order +-60, the running max moves on most tiles."""
    w = custom(1, 2, 640, 640, 128, True, seed=99, q_factor=8.0)
    q, k, v = make_qkv(w)
    o, lse = run("fa_prefill_forward", q, k, v, True, w.scale)
    ro, rl = oracle_full(q, k, v, True, w.scale)
    compare(o, lse, ro, rl)


def test_prefill_dominant_key_on_a_later_tile():
    """Key 300 (the third key tile) outweighs the rest of every row that sees it
    by about 2^11, and its V row is +-7.875. That tile's row sums lie between
    2^8 and 2^16, so the d = 128 kernel keeps the reference and divides O by the
    sum of the bf16 weights P V used: O is then within half a bf16 ulp of the
    exact result plus 8e-3. Dividing by the fp32 sum instead leaves the dominant
    weight's bf16 rounding (up to 2^-9 of |v|) in O: 2.8e-2 beyond half an ulp
    in a CPU model of the kernel's arithmetic. |O| near 7.6 puts the bf16
    output's own rounding at up to 1.56e-2, hence the per-element bound."""
    g = torch.Generator().manual_seed(7)
    B, H, S, d = 1, 2, 640, 128
    q = torch.randn(B, H, S, d, generator=g) * 0.25
    q[..., 0] = 8.0
    k = torch.randn(B, H, S, d, generator=g)
    v = torch.randn(B, H, S, d, generator=g)
    k[:, :, 300, 0] = 13.25
    v[:, :, 300, :] = torch.where(torch.arange(d) % 2 == 0, 7.875, -7.875)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o, lse = run("fa_prefill_forward", q, k, v, True, scale)
    ro, rl = oracle_full(q, k, v, True, scale)
    og = np.asarray(o, dtype=np.float64)
    ro = np.asarray(ro, dtype=np.float64).reshape(og.shape)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ro), 2.0**-126))) - 8)
    excess = np.abs(og - ro) - half_ulp
    assert excess.max() <= 8e-3, excess.max()
    assert np.abs(ro[0, :, 300:]).max() > 7.0  # the dominant key decides the rows that see it
    lg = np.asarray(lse, dtype=np.float64)
    assert np.abs(lg - np.asarray(rl, dtype=np.float64).reshape(lg.shape)).max() <= 1e-3


def test_prefill_matches_simt_reference():
    w = custom(2, 2, 384, 512, 128, True, seed=5)
    q, k, v = make_qkv(w)
    o1, l1 = run("fa_prefill_forward", q, k, v, True, w.scale)
    o2, l2 = run("fa_reference_forward_simt", q, k, v, True, w.scale)
    assert (o1 - o2).abs().max().item() < 2e-2
    assert (l1 - l2).abs().max().item() < 1e-3


# ---------------------------------------------------------------- persistent scheduling
def _prefill_dev(w, q, k, v, stream=None):
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=q.device)
    _capi.check(_capi.fa_prefill_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal,
                                         w.scale, stream), "fa_prefill_forward")
    return o, lse


@pytest.mark.parametrize("shape", [(2, 74, 1024, True), (1, 4, 2048, True), (1, 3, 700, False)])
def test_prefill_item_order_does_not_change_results(shape):
    """The persistent kernel hands items to CTAs in whatever order they free up
    (heaviest-first groups for short causal problems): every launch gives the
    same bits, and they agree with the oracle on sampled rows."""
    B, H, S, causal = shape
    w = custom(B, H, S, S, 128, causal, seed=21)
    q, k, v = (t.cuda() for t in make_qkv(w))
    o1, l1 = _prefill_dev(w, q, k, v)
    for _ in range(3):
        o2, l2 = _prefill_dev(w, q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rows = sample_rows(w, n_total=48)
    ro, rl = oracle_rows(*(t.cpu() for t in (q, k, v)), causal, w.scale, rows)
    og, lg = gather_rows(o1.float().cpu(), l1.cpu(), rows)
    compare(og, lg, ro, rl)


def test_prefill_concurrent_launches_on_separate_streams():
    """Launches in flight together take different work counters."""
    shapes = [custom(1, 8, 1536, 1536, 128, True, seed=31), custom(2, 4, 1000, 1000, 64, True, seed=32),
              custom(1, 6, 2048, 2048, 128, False, seed=33)]
    data = [tuple(t.cuda() for t in make_qkv(w)) for w in shapes]
    ref = [_prefill_dev(w, *d) for w, d in zip(shapes, data)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in shapes]
    for _ in range(3):
        outs = []
        for w, d, st in zip(shapes, data, streams):
            with torch.cuda.stream(st):
                outs.append(_prefill_dev(w, *d, stream=st))
        torch.cuda.synchronize()
        for (o, l), (ro, rl) in zip(outs, ref):
            assert torch.equal(o, ro) and torch.equal(l, rl)
    assert _capi.fa_device_status() == _capi.FA_OK


def test_prefill_work_counters_wrap_around():
    """More launches than counter slots: each launch returns its counter to zero."""
    w = WORKLOADS["tiny_b1h1s256d64_causal"]
    q, k, v = (t.cuda() for t in make_qkv(w))
    o0, l0 = _prefill_dev(w, q, k, v)
    o = torch.empty_like(o0)
    lse = torch.empty_like(l0)
    for _ in range(1100):
        _capi.check(_capi.fa_prefill_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, True,
                                             w.scale), "fa_prefill_forward")
    torch.cuda.synchronize()
    assert torch.equal(o, o0) and torch.equal(lse, l0)
    assert _capi.fa_device_status() == _capi.FA_OK


def test_prefill_cuda_graph_replay():
    """A captured launch replays correctly (its counter is back at zero after each run)."""
    w = custom(1, 4, 1024, 1024, 128, True, seed=41)
    q, k, v = (t.cuda() for t in make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # warm-up (sets the kernel attributes) before capture
        _capi.check(_capi.fa_prefill_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, True,
                                             w.scale, s), "warm-up")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _capi.check(_capi.fa_prefill_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, True,
                                             w.scale, s), "capture")
    for seed in (42, 43, 44):
        wn = with_seed(w, seed)
        qn, kn, vn = make_qkv(wn)
        q.copy_(qn); k.copy_(kn); v.copy_(vn)
        g.replay()
        torch.cuda.synchronize()
        ro, rl = _prefill_dev(w, q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl)


# ---------------------------------------------------------------- split-KV (verify) kernel
VERIFY_CASES = [
    # B, H, Sq, Sk, d, causal
    (2, 3, 5, 1000, 128, True),
    (1, 4, 1, 777, 64, True),
    (2, 2, 16, 300, 128, False),
    (1, 2, 8, 64, 128, True),
    (1, 1, 9, 5, 128, True),       # Sk < Sq: the first rows see nothing
    (1, 2, 3, 4096, 64, False),
]


@pytest.mark.parametrize("case", VERIFY_CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
@pytest.mark.parametrize("n_split", [0, 1, 2, 3, 7, "max"])
def test_verify_split_counts(case, n_split):
    B, H, Sq, Sk, d, causal = case
    max_split = -(-Sk // 64)
    ns = max_split if n_split == "max" else n_split
    if ns > max_split:
        pytest.skip("more splits than 64-key chunks")
    w = custom(B, H, Sq, Sk, d, causal, seed=Sk + Sq, q_factor=2.0)
    q, k, v = make_qkv(w)
    o, lse = run("fa_verify_forward", q, k, v, causal, w.scale, n_split=ns)
    ro, rl = oracle_full(q, k, v, causal, w.scale)
    compare(o, lse, ro, rl)


def test_verify_rejects_small_workspace():
    w = custom(1, 2, 5, 1024, 128, True)
    q, k, v = (t.cuda() for t in make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 5, dtype=torch.float32, device="cuda")
    need = _capi.fa_verify_workspace_size(1, 2, 5, 1024, 128, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = _capi.fa_verify_forward(q, k, v, o, lse, 1, 2, 5, 1024, 128, 1, w.scale, 4, ws, need - 1)
    assert st == _capi.FA_ERR_WORKSPACE
    st = _capi.fa_verify_forward(q, k, v, o, lse, 1, 2, 5, 1024, 128, 1, w.scale, 4, None, 0)
    assert st == _capi.FA_ERR_WORKSPACE


@pytest.mark.parametrize("entry", ["fa_forward", "fa_forward_ws"])
@pytest.mark.parametrize("Sq", [1, 5, 16, 17])
def test_dispatch_entry_points(entry, Sq):
    w = custom(2, 2, Sq, 700, 128, True, seed=Sq)
    q, k, v = make_qkv(w)
    o, lse = run(entry, q, k, v, True, w.scale)
    ro, rl = oracle_full(q, k, v, True, w.scale)
    compare(o, lse, ro, rl)


# ---------------------------------------------------------------- host-resident tensors
@pytest.mark.parametrize("case", [(2, 3, 300, 300, 128, True), (1, 5, 5, 1000, 128, True),
                                  (2, 2, 129, 700, 64, False), (1, 1, 3, 64, 64, True)],
                         ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("own_workspace", [True, False])
def test_forward_host_buffers(case, pinned, own_workspace):
    """fa_forward_host: host inputs and outputs, transfers pipelined inside the call."""
    B, H, Sq, Sk, d, causal = case
    w = custom(B, H, Sq, Sk, d, causal, seed=Sq + 7 * Sk)
    q, k, v = make_qkv(w)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o = torch.full((B, H, Sq, d), float("nan"), dtype=torch.bfloat16, pin_memory=pinned)
    lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, pin_memory=pinned)
    ws, ws_bytes = None, 0
    if own_workspace:
        ws_bytes = _capi.fa_forward_host_workspace_size(B, H, Sq, Sk, d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    _capi.check(_capi.fa_forward_host(q, k, v, o, lse, B, H, Sq, Sk, d, causal, w.scale, ws,
                                      ws_bytes), "fa_forward_host")
    torch.cuda.current_stream().synchronize()
    _capi.check(_capi.fa_device_status(), "device status")
    ro, rl = oracle_full(q, k, v, causal, w.scale)
    compare(o.float(), lse, ro, rl)


def test_forward_host_output_paths_agree_bit_for_bit():
    """O returns through stores by a few CTAs into a pinned, 16-byte aligned host
    buffer, and through cudaMemcpyAsync into a pageable or unaligned one: the
    bytes are the same."""
    B, H, S, d = 2, 4, 640, 128
    w = custom(B, H, S, S, d, True, seed=5)
    q, k, v = (t.pin_memory() for t in make_qkv(w))
    n = q.numel()
    outs = []
    for kind in ("pinned", "pageable", "pinned_unaligned"):
        if kind == "pinned":
            o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, pin_memory=True)
        elif kind == "pageable":
            o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16)
        else:
            base = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, pin_memory=True)
            o = base[1:1 + n].view(q.shape)  # 2 bytes past a 16-byte boundary
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32)
        _capi.check(_capi.fa_forward_host(q, k, v, o, lse, B, H, S, S, d, True, w.scale, None, 0),
                    "fa_forward_host")
        torch.cuda.current_stream().synchronize()
        _capi.check(_capi.fa_device_status(), "device status")
        outs.append((o.clone(), lse.clone()))
    assert torch.isfinite(outs[0][0].float()).all()
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_forward_host_rejects_a_small_workspace():
    w = custom(1, 2, 300, 300, 128, True)
    q, k, v = make_qkv(w)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 300)
    need = _capi.fa_forward_host_workspace_size(1, 2, 300, 300, 128)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert _capi.fa_forward_host(q, k, v, o, lse, 1, 2, 300, 300, 128, 1, w.scale, ws,
                                 need - 1) == _capi.FA_ERR_WORKSPACE


# ---------------------------------------------------------------- the pages' workloads
def test_verify_workload_full():
    """B=16, H=32, Sq=5 after a 4091-token cache (query i sees keys [0, 4091+i]), every row."""
    w = WORKLOADS["verify_b16h32q5k4096d128"]
    q, k, v = make_qkv(w)
    o, lse = run("fa_forward", q, k, v, w.causal, w.scale)
    ro, rl = oracle_full(q, k, v, w.causal, w.scale)
    compare(o, lse, ro, rl)


@pytest.mark.parametrize("name", ["prefill_b4h32s2048d128_causal", "prefill_b4h32s2048d128_causal_q4"])
def test_prefill_2k_workloads_full(name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w)
    o, lse = run("fa_forward", q, k, v, w.causal, w.scale)
    ro, rl = oracle_full(q, k, v, w.causal, w.scale)
    compare(o, lse, ro, rl)


def test_prefill_8k_headline_sampled_rows():
    """The headline workload in its timed configuration; 64 seeded (b, h, i) rows."""
    w = WORKLOADS["prefill_b4h32s8192d128_causal"]
    q, k, v = make_qkv(w)
    o, lse = run("fa_forward", q, k, v, w.causal, w.scale)
    rows = sample_rows(w, n_total=64)
    ro, rl = oracle_rows(q, k, v, w.causal, w.scale, rows)
    go, gl = gather_rows(o, lse, rows)
    compare(go, gl, ro, rl)
    # the row every causal prefill pins: query 0 attends to key 0 only
    assert torch.allclose(o[:, :, 0], v[:, :, 0].float(), atol=0, rtol=0)


def test_prefill_32k_d64_sampled_rows():
    """B=1, H=32, S=32768, d=64; 64 rows per head incl. first, last and tile boundaries."""
    w = WORKLOADS["prefill_b1h32s32768d64_causal"]
    q, k, v = make_qkv(w)
    o, lse = run("fa_forward", q, k, v, w.causal, w.scale)
    rows = sample_rows(w, per_head=64)
    ro, rl = oracle_rows(q, k, v, w.causal, w.scale, rows)
    go, gl = gather_rows(o, lse, rows)
    compare(go, gl, ro, rl)
