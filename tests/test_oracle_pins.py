"""Pins for the fp64 oracle: facts the pages and the mathematics fix.

None of these compares the oracle with a retyping of its own formula. They
check invariants (rows of P sum to 1, constant V, single key, permutation and
shift invariance), closed forms (zero query, causal first row), the
equivalence of the online and split forms with the two-pass definition, an
independent numpy restatement and torch's fp64 SDPA on tiny inputs, and the
hand-derived golden cases under tests/golden/.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.numpy_ref import attention_np, to_f64
from exact_tiled_attention_03_gb300.inputs import custom, make_qkv
from golden_io import hand_examples, isclose_or_both_inf

TOL = 1e-12

SHAPES = [
    # B, H, Sq, Sk, d, causal
    (1, 1, 7, 7, 16, True),
    (1, 2, 5, 13, 8, True),       # bottom-right offset, Sq < Sk
    (2, 1, 9, 4, 8, True),        # Sk < Sq: some rows fully masked
    (1, 1, 6, 11, 16, False),
    (2, 2, 17, 17, 32, False),
]


def case(B, H, Sq, Sk, d, causal, seed=0, factor=1.0):
    w = custom(B, H, Sq, Sk, d, causal, seed=seed, q_factor=factor)
    q, k, v = make_qkv(w)
    return w, q, k, v


def visible(i, Sq, Sk, causal):
    return Sk if not causal else max(0, min(Sk, i + Sk - Sq + 1))


@pytest.mark.parametrize("shape", SHAPES)
def test_probability_rows_sum_to_one(shape):
    """Softmax normalisation (Warmup Guide, Chapter 2): each visible row of P sums to 1."""
    w, q, k, v = case(*shape, seed=3, factor=3.0)
    for b in range(w.B):
        for h in range(w.H):
            for i in range(w.Sq):
                p = oracle.probs_row(q, k, w.causal, w.scale, b, h, i)
                nv = visible(i, w.Sq, w.Sk, w.causal)
                assert np.all(p >= 0)
                assert np.all(p[nv:] == 0), "hidden keys must get zero weight"
                if nv:
                    assert abs(p.sum() - 1.0) < TOL
                    assert np.all(p[:nv] > 0)
                else:
                    assert p.sum() == 0


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("c", [1.5, -3.25])
def test_constant_v_returns_the_constant(shape, c):
    """A convex combination of identical rows is that row, for every mask."""
    w, q, k, v = case(*shape, seed=5)
    v = torch.full_like(v, c)
    o, lse = oracle.attention(q, k, v, w.causal, w.scale)
    for i in range(w.Sq):
        nv = visible(i, w.Sq, w.Sk, w.causal)
        expect = c if nv else 0.0
        assert np.max(np.abs(o[:, :, i, :] - expect)) < TOL


@pytest.mark.parametrize("d", [1, 8, 64])
def test_single_key_returns_its_value_row(d):
    """Sk = 1: the only weight is 1, so o = v_0 and lse = s_0 = scale * q . k_0."""
    w, q, k, v = case(2, 3, 4, 1, d, False, seed=7)
    o, lse = oracle.attention(q, k, v, False, w.scale)
    qd, kd, vd = to_f64(q), to_f64(k), to_f64(v)
    for b in range(w.B):
        for h in range(w.H):
            for i in range(w.Sq):
                assert np.max(np.abs(o[b, h, i] - vd[b, h, 0])) == 0.0
                s0 = float(np.float32(w.scale)) * float(np.dot(qd[b, h, i], kd[b, h, 0]))
                assert abs(lse[b, h, i] - s0) < TOL * max(1.0, abs(s0))


def test_causal_first_row_is_first_value_row():
    """Sq = Sk causal: query 0 sees key 0 only (the first row of every causal prefill)."""
    w, q, k, v = case(2, 2, 33, 33, 16, True, seed=11, factor=4.0)
    o, lse = oracle.attention(q, k, v, True, w.scale, rows=[(b, h, 0) for b in range(2) for h in range(2)])
    qd, kd, vd = to_f64(q), to_f64(k), to_f64(v)
    for n, (b, h) in enumerate([(b, h) for b in range(2) for h in range(2)]):
        assert np.all(o[n] == vd[b, h, 0])
        s0 = float(np.float32(w.scale)) * float(np.dot(qd[b, h, 0], kd[b, h, 0]))
        assert abs(lse[n] - s0) < TOL * max(1.0, abs(s0))


@pytest.mark.parametrize("shape", SHAPES)
def test_zero_query_gives_prefix_means(shape):
    """Q = 0: every logit is 0, so o_i = mean of the visible v_j and lse_i = ln(#visible)."""
    w, q, k, v = case(*shape, seed=13)
    q = torch.zeros_like(q)
    o, lse = oracle.attention(q, k, v, w.causal, w.scale)
    vd = to_f64(v)
    for i in range(w.Sq):
        nv = visible(i, w.Sq, w.Sk, w.causal)
        if nv == 0:
            assert np.all(o[:, :, i] == 0) and np.all(np.isneginf(lse[:, :, i]))
            continue
        assert np.max(np.abs(o[:, :, i] - vd[:, :, :nv].mean(axis=2))) < TOL
        assert np.max(np.abs(lse[:, :, i] - math.log(nv))) < TOL


@pytest.mark.parametrize("shape", SHAPES)
def test_zero_scale_gives_visible_means_for_any_query(shape):
    """scale = 0 makes every logit 0 whatever Q is (the scale is a plain factor of
    the scores, Warmup Guide Ch.4): o_i = mean of the visible v_j, lse_i = ln(#visible)."""
    w, q, k, v = case(*shape, seed=17, factor=4.0)
    o, lse = oracle.attention(q, k, v, w.causal, 0.0)
    vd = to_f64(v)
    for i in range(w.Sq):
        nv = visible(i, w.Sq, w.Sk, w.causal)
        if nv == 0:
            assert np.all(o[:, :, i] == 0) and np.all(np.isneginf(lse[:, :, i]))
            continue
        assert np.max(np.abs(o[:, :, i] - vd[:, :, :nv].mean(axis=2))) < TOL
        assert np.max(np.abs(lse[:, :, i] - math.log(nv))) < TOL


@pytest.mark.parametrize("shape", SHAPES)
def test_negative_scale_equals_the_negated_query(shape):
    """s_j = scale * (q . k_j) is odd in scale and linear in q, so scale -c on q
    gives exactly what +c gives on -q (bf16 negation is exact). A kernel that
    takes |scale| fails this, as does one whose max ignores the sign."""
    w, q, k, v = case(*shape, seed=19)
    c = float(np.float32(w.scale))
    o1, l1 = oracle.attention(q, k, v, w.causal, -c)
    o2, l2 = oracle.attention(-q, k, v, w.causal, c)
    o3, l3 = oracle.attention(q, k, v, w.causal, c)
    assert np.max(np.abs(o1 - o2)) < TOL
    fin = np.isfinite(l2)
    assert np.array_equal(np.isfinite(l1), fin)
    assert np.max(np.abs(l1[fin] - l2[fin]), initial=0.0) < TOL
    assert np.max(np.abs(o1 - o3)) > 1e-3   # the sign really matters on these inputs


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_online_forms_equal_two_pass(form, causal):
    """Online softmax block accumulation equals the two-pass result for any block size
    (page 1 Mechanics pseudocode = form 1; Warmup Guide Chapter 3 = form 2; Lab 01's
    per-block rescaling check). Q x 4 makes the running max move often."""
    Sk = 300
    w, q, k, v = case(1, 2, 37, Sk, 16, causal, seed=17, factor=4.0)
    o2, l2 = oracle.attention(q, k, v, causal, w.scale)
    o2 = o2.reshape(-1, 16)
    l2 = l2.reshape(-1)
    for block in [1, 7, 64, 128, 129, Sk]:
        o1, l1 = oracle.online(q, k, v, causal, w.scale, block, form)
        assert np.max(np.abs(o1 - o2)) < TOL, block
        assert np.max(np.abs(l1 - l2)) < TOL, block


def test_online_forms_on_a_one_dimensional_toy():
    """Lab 01's 1-D toy: d = 1, a single query, logits spanning +-40, every block size."""
    torch.manual_seed(0)
    w, q, k, v = case(1, 1, 1, 50, 1, False, seed=19)
    q = torch.tensor([[[[8.0]]]], dtype=torch.bfloat16)
    o2, l2 = oracle.attention(q, k, v, False, 1.0)
    for block in range(1, 51):
        for form in (1, 2):
            o1, l1 = oracle.online(q, k, v, False, 1.0, block, form)
            assert abs(o1[0, 0] - o2[0, 0, 0, 0]) < TOL
            assert abs(l1[0] - l2[0, 0, 0]) < TOL


@pytest.mark.parametrize("causal", [False, True])
def test_split_combine_equals_unsplit(causal):
    """Flash-Decoding's split + final combine (Lecture 06, section 5) reproduces the
    unsplit result for any partition of the keys, empty chunks included."""
    Sk = 200
    w, q, k, v = case(2, 2, 5, Sk, 32, causal, seed=23, factor=2.0)
    o_ref, l_ref = oracle.attention(q, k, v, causal, w.scale)
    o_ref = o_ref.reshape(-1, 32)
    l_ref = l_ref.reshape(-1)
    g = np.random.default_rng(0)
    partitions = [[0, Sk], [0, 100, Sk], [0, 0, 50, 50, Sk], [0, 199, Sk], [0, 196, 197, Sk]]
    for _ in range(5):
        cuts = sorted(g.choice(np.arange(1, Sk), size=g.integers(1, 9), replace=False).tolist())
        partitions.append([0] + cuts + [Sk])
    for bounds in partitions:
        o, l = oracle.split(q, k, v, causal, w.scale, bounds)
        assert np.max(np.abs(o - o_ref)) < TOL, bounds
        assert np.max(np.abs(l - l_ref)) < TOL, bounds


def test_combine_of_separately_computed_parts_equals_unsplit():
    """Partials computed as independent attention problems over disjoint key ranges
    (non-causal parts, and the final part with its own bottom-right causal offset)
    combine to the unsplit causal result."""
    Sk, Sq = 300, 5
    w, q, k, v = case(1, 3, Sq, Sk, 16, True, seed=43, factor=3.0)
    o_ref, l_ref = oracle.attention(q, k, v, True, w.scale)
    cut = 180  # every query sees keys [0, 295 + i], so [0, 180) is fully visible
    o_a, l_a = oracle.attention(q, k[:, :, :cut], v[:, :, :cut], False, w.scale)
    o_b, l_b = oracle.attention(q, k[:, :, cut:], v[:, :, cut:], True, w.scale)
    o, l = oracle.combine(np.stack([o_a.reshape(-1, 16), o_b.reshape(-1, 16)]),
                          np.stack([l_a.reshape(-1), l_b.reshape(-1)]))
    assert np.max(np.abs(o - o_ref.reshape(-1, 16))) < TOL
    assert np.max(np.abs(l - l_ref.reshape(-1))) < TOL
    # an empty part (lse = -inf) has no weight
    o2, l2 = oracle.combine(np.stack([o_a.reshape(-1, 16), np.zeros((15, 16))]),
                            np.stack([l_a.reshape(-1), np.full(15, -np.inf)]))
    assert np.array_equal(o2, o_a.reshape(-1, 16)) and np.array_equal(l2, l_a.reshape(-1))


def _causal_visible(B, Sq, Sk):
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    return np.broadcast_to(j <= i + (Sk - Sq), (B, Sq, Sk)).astype(np.uint8)


@pytest.mark.parametrize("shape", SHAPES)
def test_masked_definition_reduces_to_causal_and_full(shape):
    """An all-ones mask is non-causal attention; the bottom-right triangle is causal."""
    B, H, Sq, Sk, d, causal = shape
    w, q, k, v = case(B, H, Sq, Sk, d, causal, seed=47, factor=2.0)
    o_full, l_full = oracle.attention(q, k, v, False, w.scale)
    o, l = oracle.attention_masked(q, k, v, np.ones((B, Sq, Sk), np.uint8), w.scale)
    assert np.max(np.abs(o - o_full)) < TOL and np.max(np.abs(l - l_full)) < TOL
    o_c, l_c = oracle.attention(q, k, v, True, w.scale)
    o, l = oracle.attention_masked(q, k, v, _causal_visible(B, Sq, Sk), w.scale)
    assert np.max(np.abs(o - o_c)) < TOL
    fin = np.isfinite(l_c)
    assert np.array_equal(fin, np.isfinite(l)) and np.max(np.abs(l[fin] - l_c[fin])) < TOL


def test_masked_definition_single_key_and_subset_equivalence():
    """A row that sees one key returns its value row; a row that sees a key subset equals
    plain attention over that subset of keys (a gather of K and V)."""
    w, q, k, v = case(2, 2, 4, 12, 16, False, seed=53, factor=3.0)
    vis = np.zeros((2, 4, 12), np.uint8)
    vis[:, 0, 7] = 1                               # row 0: key 7 only
    vis[:, 1, [0, 3, 5, 11]] = 1                   # row 1: a scattered subset
    vis[:, 2, :] = 1                               # row 2: everything
    o, l = oracle.attention_masked(q, k, v, vis, w.scale)   # row 3: nothing
    vd = to_f64(v)
    assert np.all(o[:, :, 0] == vd[:, :, 7])
    sub = [0, 3, 5, 11]
    o_s, l_s = oracle.attention(q[:, :, 1:2], k[:, :, sub], v[:, :, sub], False, w.scale)
    assert np.max(np.abs(o[:, :, 1] - o_s[:, :, 0])) < TOL
    assert np.max(np.abs(l[:, :, 1] - l_s[:, :, 0])) < TOL
    o_f, l_f = oracle.attention(q[:, :, 2:3], k, v, False, w.scale)
    assert np.max(np.abs(o[:, :, 2] - o_f[:, :, 0])) < TOL
    assert np.all(o[:, :, 3] == 0) and np.all(np.isneginf(l[:, :, 3]))


def test_key_value_permutation_invariance():
    """Non-causal attention is a function of the set of (key, value) pairs."""
    w, q, k, v = case(1, 2, 9, 40, 16, False, seed=29)
    o, l = oracle.attention(q, k, v, False, w.scale)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(1))
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], False, w.scale)
    assert np.max(np.abs(o - o2)) < TOL and np.max(np.abs(l - l2)) < TOL


def test_shift_of_all_keys_shifts_lse_only():
    """Adding u to every key adds scale*q.u to every logit of row i: P and O are
    unchanged (the safe softmax's shift identity, Chapter 2) and lse moves by scale*q.u."""
    g = torch.Generator().manual_seed(31)
    q = torch.randint(-3, 4, (1, 1, 6, 8), generator=g).to(torch.bfloat16)
    k = torch.randint(-3, 4, (1, 1, 10, 8), generator=g).to(torch.bfloat16)
    v = torch.randn((1, 1, 10, 8), generator=g).to(torch.bfloat16)
    u = torch.randint(-2, 3, (8,), generator=g).to(torch.bfloat16)
    scale = 0.25
    for causal in (False, True):
        o, l = oracle.attention(q, k, v, causal, scale)
        o2, l2 = oracle.attention(q, k + u, v, causal, scale)
        shift = scale * (to_f64(q)[0, 0] @ to_f64(u))
        assert np.max(np.abs(o - o2)) < 1e-12
        assert np.max(np.abs(l2[0, 0] - (l[0, 0] + shift))) < 1e-12


@pytest.mark.parametrize("shape", SHAPES + [(1, 1, 64, 64, 64, True), (1, 1, 1, 130, 128, True)])
def test_matches_independent_numpy_restatement(shape):
    w, q, k, v = case(*shape, seed=37, factor=2.0)
    o, lse = oracle.attention(q, k, v, w.causal, w.scale)
    on, ln = attention_np(to_f64(q), to_f64(k), to_f64(v), w.causal, w.scale)
    assert np.max(np.abs(o - on)) < TOL
    fin = np.isfinite(ln)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - ln[fin]), initial=0.0) < TOL


@pytest.mark.parametrize("sign", [1.0, 0.0, -1.0])
@pytest.mark.parametrize("shape", [s for s in SHAPES if s[2] <= s[3] or not s[5]])
def test_matches_torch_sdpa_fp64(shape, sign):
    """torch.nn.functional.scaled_dot_product_attention (CPU, fp64, math path) with an
    explicit bottom-right mask; lse from torch.logsumexp of the masked logits. The
    scale is 1/sqrt(d), 0 or -1/sqrt(d)."""
    w, q, k, v = case(*shape, seed=41)
    scale = float(np.float32(w.scale)) * sign
    o, lse = oracle.attention(q, k, v, w.causal, scale)
    qd, kd, vd = q.double(), k.double(), v.double()
    mask = None
    if w.causal:
        i = torch.arange(w.Sq)[:, None]
        j = torch.arange(w.Sk)[None, :]
        mask = j <= i + (w.Sk - w.Sq)
    sc = scale
    ot = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=sc)
    logits = sc * (qd @ kd.transpose(-1, -2))
    if mask is not None:
        logits = logits.masked_fill(~mask, float("-inf"))
    lt = torch.logsumexp(logits, dim=-1)
    assert np.max(np.abs(o - ot.numpy())) < 1e-12
    assert np.max(np.abs(lse - lt.numpy())) < 1e-12


@pytest.mark.parametrize("c", hand_examples(), ids=lambda c: c["name"])
def test_hand_derived_golden_cases(c):
    shape4 = lambda m, S: torch.tensor(m, dtype=torch.float64).reshape(c["B"], c["H"], S, c["d"])
    q = shape4(c["q"], c["Sq"])
    k = shape4(c["k"], c["Sk"])
    v = shape4(c["v"], c["Sk"])
    for t in (q, k, v):   # fixtures must be exact in bf16
        assert torch.equal(t.to(torch.bfloat16).double(), t)
    o, lse = oracle.attention(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
                              c["causal"], c["scale"])
    expect_o = np.asarray(c["o"], dtype=np.float64).reshape(o.shape)
    assert np.max(np.abs(o - expect_o)) <= c["tol"], c["cite"]
    for got, exp in zip(lse.reshape(-1), c["lse"]):
        assert isclose_or_both_inf(float(got), exp, c["tol"]), c["cite"]
