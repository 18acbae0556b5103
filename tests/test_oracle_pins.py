"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test is chosen so that a plausible mistake in the oracle (a dropped
ReLU, a wrong sign in the sigmoid, a transposed operand, a wrong index in the
neuron table, a non-strict candidate test, an off-by-one in the bit layout)
fails at least one of them. The pins are: hand-derived closed forms
(tests/golden/closed_form_cases.json), the all-active special case against a
library dense FFN (torch.nn.functional in float64), brute force on d=8,
f=32/64, invariants (disjoint-mask linearity, permutation invariance) and the
closed form of the momentum recursion.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import sffn_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as fh:
        return json.load(fh)


# ---------------------------------------------------------------- predictor

def _pred_case(g):
    p = g["predictor"]
    W1 = np.array(p["W1"], dtype=np.float64)
    x = np.array(p["x"], dtype=np.float64)
    W2 = np.array([[i - 16, 7, -1] for i in range(p["f"])], dtype=np.float64)
    return p, W1, x, W2


def test_predictor_closed_form(golden):
    p, W1, x, W2 = _pred_case(golden)
    hid = O.predictor_hidden(W1, x)
    assert hid.tolist() == p["cases"][0]["hid"]
    scores = O.predictor_scores(W2, hid)
    assert scores.tolist() == [2.0 * i - 36.5 for i in range(p["f"])]
    for case in p["cases"]:
        act = O.active_from_scores(scores, case["thres"])
        v = O.mask_views(act, p["group_size"])
        assert v["count"] == case["count"]
        assert v["nmask"].tolist() == case["nmask"]
        assert v["gmask"].tolist() == case["gmask"]
        first = int(v["idx"][0]) if v["count"] else None
        assert first == case["first_idx"]
        assert v["idx"].tolist() == sorted(v["idx"].tolist())


def test_predictor_biases_shift_scores():
    # b1 enters before the ReLU, b2 after: with W1 = I, x = [-1, 2], b1 = [3, -5]:
    # pre = [2, -3] -> hid = [2, 0]; W2 = [[1, 1]], b2 = [-2.5] -> s = -0.5.
    W1 = np.eye(2)
    hid = O.predictor_hidden(W1, np.array([-1.0, 2.0]), np.array([3.0, -5.0]))
    assert hid.tolist() == [2.0, 0.0]
    s = O.predictor_scores(np.array([[1.0, 1.0]]), hid, np.array([-2.5]))
    assert s.tolist() == [-0.5]


def test_threshold_nan_and_equality():
    s = np.array([0.0, -0.0, np.nan, 1e-300, -1e-300, np.inf, -np.inf])
    assert O.active_from_scores(s, 0.0).tolist() == [True, True, False, True, False, True, False]


def test_bit_layout_roundtrip():
    rng = np.random.default_rng(1)
    for f in (32, 64, 96, 2048):
        bits = rng.random(f) < 0.3
        w = O.bits_to_words(bits)
        assert w.shape == (f // 32,)
        assert (O.words_to_bits(w, f) == bits).all()
        # bit i%32 of word i//32, checked against python ints
        for i in np.flatnonzero(bits)[:20]:
            assert (int(w[i // 32]) >> (i % 32)) & 1 == 1
    assert O.bits_to_words(np.array([True] + [False] * 30 + [True])).tolist() == [0x80000001]


def test_group_mask_size_64():
    act = np.zeros(256, dtype=bool)
    act[[70, 255]] = True          # group 1 (64..127) and group 3 (192..255)
    v = O.mask_views(act, 64)
    assert v["gmask"].tolist() == [0b1010]
    assert v["nmask"].tolist() == [0, 0, 1 << 6, 0, 0, 0, 0, 1 << 31]


# ---------------------------------------------------------------- FFN closed forms

def test_ffn_reglu_closed_form(golden):
    c = golden["ffn_reglu"]
    f, d = c["f"], c["d"]
    up = np.zeros((f, d))
    gate = np.zeros((f, d))
    down = np.zeros((d, f))
    for i in range(f):
        up[i] = [100.0, (i - 4) / 2.0, -100.0]
        gate[i] = [-100.0, (i % 3) - 1.0, 100.0]
        down[:, i] = [1.0, i, -i]
    act = np.zeros(f, dtype=bool)
    act[c["active_slots"]] = True
    y, h = O.ffn_sparse(np.array(c["x"], dtype=np.float64), up, gate, down, "reglu", act)
    assert y.tolist() == c["y"]
    assert h.tolist() == [0, 0, -1, 0, 0, 0.5, 0, 0, 2, 0, 0, 3.5]


def test_ffn_swiglu_relu_closed_form(golden):
    want = golden["ffn_swiglu"]["h_for_g_ln3_u4"]
    h = O.activation("swiglu", np.array([4.0, 7.0]), np.array([math.log(3.0), 0.0]))
    assert abs(h[0] - want) < 1e-15 and h[1] == 0.0
    # SiLU is odd-symmetric around its linear part: SiLU(g) - SiLU(-g) = g
    g = np.linspace(-6, 6, 13)
    one = np.ones_like(g)
    assert np.allclose(O.activation("swiglu", one, g) - O.activation("swiglu", one, -g), g, atol=1e-14)
    assert O.activation("relu", np.array([-2.0, 3.0]), None).tolist() == [0.0, 3.0]
    assert O.activation("relu2", np.array([-2.0, 3.0, 0.5]), None).tolist() == [0.0, 9.0, 0.25]
    assert O.activation("reglu", np.array([5.0, 5.0]), np.array([-1.0, 2.0])).tolist() == [0.0, 10.0]


# ---------------------------------------------------------------- library special case

def _rand_layer(rng, d, f, act):
    up = rng.standard_normal((f, d))
    gate = rng.standard_normal((f, d)) if act in ("reglu", "swiglu") else None
    down = rng.standard_normal((d, f))
    return up, gate, down


def _torch_dense(x, up, gate, down, act):
    xt = torch.from_numpy(x)
    u = F.linear(xt, torch.from_numpy(up))
    if act == "relu":
        h = F.relu(u)
    elif act == "relu2":
        h = torch.square(F.relu(u))
    elif act == "reglu":
        h = F.relu(F.linear(xt, torch.from_numpy(gate))) * u
    else:
        h = F.silu(F.linear(xt, torch.from_numpy(gate))) * u
    return F.linear(h, torch.from_numpy(down)).numpy()


@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu", "relu2"])
def test_all_active_equals_library_dense(act):
    rng = np.random.default_rng(7)
    d, f, h = 24, 64, 16
    up, gate, down = _rand_layer(rng, d, f, act)
    W1 = rng.standard_normal((h, d))
    W2 = rng.standard_normal((f, h))
    perm = rng.permutation(f)
    x = rng.standard_normal(d)
    r = O.decode_layer(x, W1, W2, up, gate, down, act, -np.inf, 32, perm=perm)
    assert r["count"] == f
    ref = _torch_dense(x, up, gate, down, act)
    assert np.allclose(r["y"], ref, rtol=1e-12, atol=1e-12)
    # predictor against the library too
    hid = F.relu(F.linear(torch.from_numpy(x), torch.from_numpy(W1)))
    s = F.linear(hid, torch.from_numpy(W2)).numpy()
    assert np.allclose(r["scores"], s[perm], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu", "relu2"])
def test_none_active_is_exact_zero(act):
    rng = np.random.default_rng(8)
    d, f, h = 16, 64, 8
    up, gate, down = _rand_layer(rng, d, f, act)
    r = O.decode_layer(rng.standard_normal(d), rng.standard_normal((h, d)), rng.standard_normal((f, h)),
                       up, gate, down, act, np.inf, 32)
    assert r["count"] == 0 and not r["nmask"].any() and not r["gmask"].any()
    assert (r["y"] == 0.0).all() and r["y"].shape == (d,)


# ---------------------------------------------------------------- brute force d=8

@pytest.mark.parametrize("f", [32, 64])
@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu", "relu2"])
def test_brute_force_masks_d8(f, act):
    """For random masks, y equals the library dense FFN with the inactive
    neurons' up/gate rows and down columns zeroed; disjoint masks add."""
    rng = np.random.default_rng(100 + f)
    d = 8
    up, gate, down = _rand_layer(rng, d, f, act)
    perm = rng.permutation(f)
    x = rng.standard_normal(d)
    for trial in range(1000 if act == "relu" else 300):
        act_slots = rng.random(f) < rng.random()
        y, _ = O.ffn_sparse(x, up, gate, down, act, act_slots, perm)
        keep = np.zeros(f, dtype=bool)
        keep[perm[act_slots]] = True            # original ids of the active slots
        upz = up * keep[:, None]
        gz = gate * keep[:, None] if gate is not None else None
        dz = down * keep[None, :]
        ref = _torch_dense(x, upz, gz, dz, act)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12), trial
        if trial < 50:
            other = (~act_slots) & (rng.random(f) < 0.5)
            y2, _ = O.ffn_sparse(x, up, gate, down, act, other, perm)
            y12, _ = O.ffn_sparse(x, up, gate, down, act, act_slots | other, perm)
            assert np.allclose(y12, y + y2, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- zero-skip

def test_zero_skip_hand_computed():
    """d = 2, f = 4, x = (1, 2); h and y worked out by hand."""
    x = np.array([1.0, 2.0])
    down = np.array([[1.0, 2.0, 3.0, 4.0], [5.0, 6.0, 7.0, 8.0]])
    up = np.array([[1.0, 0.0], [-1.0, 0.0], [0.0, 0.0], [1.0, 1.0]])       # u = (1, -1, 0, 3)
    allon = np.ones(4, dtype=bool)
    y, n = O.ffn_sparse_zero_skip(x, up, None, down, "relu", allon)       # h = (1, 0, 0, 3)
    assert n == 2 and np.array_equal(y, [1 + 12, 5 + 24])
    y, n = O.ffn_sparse_zero_skip(x, up, None, down, "relu2", allon)      # h = (1, 0, 0, 9)
    assert n == 2 and np.array_equal(y, [1 + 36, 5 + 72])
    # slots 0, 2, 3 active: h = (1, 0, 3) -> two columns
    y, n = O.ffn_sparse_zero_skip(x, up, None, down, "relu", np.array([True, False, True, True]))
    assert n == 2 and np.array_equal(y, [13, 29])
    # ReGLU: g = (-1, 1, 3, -2), u = (2, 5, -1, 4) -> h = (0, 5, -3, 0)
    gate = np.array([[-1.0, 0.0], [1.0, 0.0], [1.0, 1.0], [0.0, -1.0]])
    upg = np.array([[2.0, 0.0], [5.0, 0.0], [1.0, -1.0], [0.0, 2.0]])
    y, n = O.ffn_sparse_zero_skip(x, upg, gate, down, "reglu", allon)
    assert n == 2 and np.array_equal(y, [5 * 2 - 3 * 3, 5 * 6 - 3 * 7])
    # SwiGLU is zero only where g = 0 or u = 0: g = (0, 1, 3, -2) -> h_0 = 0
    gate0 = np.array([[0.0, 0.0], [1.0, 0.0], [1.0, 1.0], [0.0, -1.0]])
    _, n = O.ffn_sparse_zero_skip(x, upg, gate0, down, "swiglu", allon)
    assert n == 3


@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu", "relu2"])
def test_zero_skip_equals_full_and_library(act):
    """Skipping the down columns of zero activations leaves y as the library
    dense FFN over the active neurons gives it, and the number of columns
    read is the library's count of non-zero activations among them."""
    rng = np.random.default_rng(300)
    d, f = 8, 64
    up, gate, down = _rand_layer(rng, d, f, act)
    perm = rng.permutation(f)
    for trial in range(200):
        x = rng.standard_normal(d)
        act_slots = rng.random(f) < rng.random()
        y, n = O.ffn_sparse_zero_skip(x, up, gate, down, act, act_slots, perm)
        keep = np.zeros(f, dtype=bool)
        keep[perm[act_slots]] = True
        upz = up * keep[:, None]
        gz = gate * keep[:, None] if gate is not None else None
        assert np.allclose(y, _torch_dense(x, upz, gz, down * keep[None, :], act), rtol=1e-12, atol=1e-12), trial
        ident = np.eye(f)
        h = _torch_dense(x, upz, gz, ident, act)      # down = identity: the library's h in original order
        assert n == int(np.count_nonzero(h[keep])), trial


def test_brute_force_scalar_predictor_d8():
    """Each a_i against a scalar recomputation in plain python floats."""
    rng = np.random.default_rng(3)
    d, h, f = 8, 4, 64
    W1 = rng.standard_normal((h, d))
    W2 = rng.standard_normal((f, h))
    b2 = rng.standard_normal(f) * 0.1
    perm = rng.permutation(f)
    for _ in range(200):
        x = rng.standard_normal(d)
        r = O.decode_layer(x, W1, W2, np.zeros((f, d)), None, np.zeros((d, f)), "relu", 0.05, 32,
                           perm=perm, b2=b2)
        for slot in range(f):
            n = perm[slot]
            hid = [max(0.0, sum(float(W1[j, k]) * float(x[k]) for k in range(d))) for j in range(h)]
            s = sum(float(W2[n, j]) * hid[j] for j in range(h)) + float(b2[n])
            if abs(s - 0.05) > 1e-9:
                assert bool(r["active"][slot]) == (s >= 0.05)


def test_permutation_invariance():
    """Re-ordering the packed slots (a different neuron table) leaves y and the
    set of active ORIGINAL neurons unchanged."""
    rng = np.random.default_rng(11)
    d, f, h = 16, 128, 8
    up, gate, down = _rand_layer(rng, d, f, "reglu")
    W1 = rng.standard_normal((h, d))
    W2 = rng.standard_normal((f, h))
    x = rng.standard_normal(d)
    p1 = rng.permutation(f)
    p2 = rng.permutation(f)
    r1 = O.decode_layer(x, W1, W2, up, gate, down, "reglu", 0.0, 32, perm=p1)
    r2 = O.decode_layer(x, W1, W2, up, gate, down, "reglu", 0.0, 32, perm=p2)
    assert np.allclose(r1["y"], r2["y"], rtol=1e-12, atol=1e-12)
    assert sorted(p1[r1["idx"]].tolist()) == sorted(p2[r2["idx"]].tolist())
    # and against the identity table
    r0 = O.decode_layer(x, W1, W2, up, gate, down, "reglu", 0.0, 32)
    assert sorted(r0["idx"].tolist()) == sorted(p1[r1["idx"]].tolist())


def test_widen_exact():
    v = np.array([1.0, -2.5, 3.140625, 65504.0, 2.0 ** -14], dtype=np.float32)
    assert O.widen(v.astype(np.float16), "f16").tolist() == v.astype(np.float64).tolist()
    bits = torch.tensor(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert O.widen(bits, "bf16").tolist() == torch.tensor(v).to(torch.bfloat16).double().tolist()
    # bf16 bit patterns by hand: 0x3F80 = 1.0, 0xC020 = -2.5, 0x0001 = smallest subnormal
    assert O.widen(np.array([0x3F80, 0xC020, 0x0001], dtype=np.uint16), "bf16").tolist() == [1.0, -2.5, 2.0 ** -133]


# ---------------------------------------------------------------- batch

def test_batch_union_and_identical_tokens():
    rng = np.random.default_rng(5)
    f = 128
    A = rng.random((4, f)) < 0.1
    u = O.batch_union(A, 32)
    assert (u["active"] == (A[0] | A[1] | A[2] | A[3])).all()
    for g in range(4):
        assert bool((int(u["ugmask"][0]) >> g) & 1) == bool(A[:, g * 32:(g + 1) * 32].any())
    same = np.repeat(A[:1], 5, axis=0)
    assert (O.batch_union(same, 32)["unmask"] == O.mask_views(A[0], 32)["nmask"]).all()


# ---------------------------------------------------------------- momentum

LAM, EPS = np.float32(0.9), np.float32(0.01)


def _run(seq, lam=LAM, eps=EPS):
    s = np.zeros(1, dtype=np.float32)
    tau = None
    for a in seq:
        s, tau = O.tam_scores_step(s, np.array([bool(a)]), lam, eps)
    return s[0], tau


def test_tam_isolated_hit_never_candidate(golden):
    s, tau = _run([1])
    assert s == np.float32(1) - LAM            # exactly 1 - lambda
    assert not s > tau
    # after any number of misses, a single hit from rest stays below tau
    for lam in (0.8, 0.85, 0.9, 0.95, 0.99):
        for pre in (0, 3, 50):
            s, tau = _run([0] * pre + [1] + [0] * 2, lam=np.float32(lam))
            assert not s > tau


def test_tam_two_hits_and_gap_rule(golden):
    s, tau = _run([1, 1])
    assert s > tau and abs(float(s) - 0.19) < 1e-6
    m_max = golden["tam"]["max_gap_still_candidate"]
    for m in range(0, 30):
        s, tau = _run([1] + [0] * m + [1])
        assert bool(s > tau) == (m <= m_max), m
    # the closed-form boundary: 0.1 * 0.9^(m+1) > 0.01  iff  m <= 20
    assert max(m for m in range(40) if 0.1 * 0.9 ** (m + 1) > 0.01) == m_max


def test_tam_matches_closed_form_random_sequences():
    rng = np.random.default_rng(2)
    for lam in (0.8, 0.9, 0.95, 0.99):
        for T in (1, 7, 64, 300):
            seq = rng.random(T) < 0.4
            s, _ = _run(seq, lam=np.float32(lam))
            cf = O.tam_closed_form(seq, float(np.float32(lam)))
            assert abs(float(s) - cf) < 1e-6, (lam, T)
    s, _ = _run([1] * 50)
    assert abs(float(s) - (1 - 0.9 ** 50)) < 1e-6
    # decay from a start value when nothing is active: s_T = lambda^T s_0
    s = np.array([0.7], dtype=np.float32)
    for _ in range(10):
        s, _ = O.tam_scores_step(s, np.array([False]), LAM, EPS)
    assert abs(float(s[0]) - 0.7 * 0.9 ** 10) < 1e-6


def _rank_resident(s, tau, K):
    """Brute-force definition: a candidate stays iff fewer than K candidates
    beat it, where h beats g iff s_h > s_g, or s_h == s_g and h < g."""
    n = s.shape[0]
    cand = [g for g in range(n) if s[g] > tau]
    res = set()
    for g in cand:
        beaten = sum(1 for k in cand if (s[k] > s[g]) or (s[k] == s[g] and k < g))
        if beaten < K:
            res.add(g)
    return set(cand), res


def test_tam_topk_against_rank_definition():
    rng = np.random.default_rng(9)
    for trial in range(200):
        n = int(rng.integers(1, 80))
        # few distinct values so that ties are common
        s = (rng.integers(0, 6, n) * np.float32(0.05)).astype(np.float32)
        tau = np.float32(0.11)
        K = int(rng.integers(0, n + 2))
        cand, topk = O.tam_select(s, tau, K)
        c_ref, r_ref = _rank_resident(s, tau, K)
        assert set(np.flatnonzero(cand).tolist()) == c_ref
        assert set(topk.tolist()) == r_ref
        # rank order: score descending, then index ascending
        keys = [(-float(s[g]), g) for g in topk]
        assert keys == sorted(keys)


def test_tam_update_sets():
    rng = np.random.default_rng(4)
    n = 300
    s = rng.random(n).astype(np.float32) * np.float32(0.5)
    prev = rng.random(n) < 0.3
    ga = rng.random(n) < 0.2
    for K in (0, 10, 150, n + 5):
        r = O.tam_update(s, prev, ga, LAM, EPS, K)
        res = r["resident"]
        assert (r["load"] == (res & ~prev)).all() and (r["evict"] == (prev & ~res)).all()
        assert (r["changed"] == (r["load"] | r["evict"])).all()
        assert ((r["load"] | (prev & res)) == res).all()
        assert not (res & ~r["cand"]).any()
        if K >= r["n_cand"]:
            assert (res == r["cand"]).all()
        if K == 0:
            assert not res.any()


def test_anb_step_clamps_and_moves():
    lam = np.float32(0.9)
    for _ in range(20):
        lam = O.anb_step(lam, True, 0.01, 0.8, 0.99)
    assert lam == np.float32(0.99)
    for _ in range(30):
        lam = O.anb_step(lam, False, 0.01, 0.8, 0.99)
    assert lam == np.float32(0.8)
    lam = O.anb_step(np.float32(0.9), True, 0.01, 0.8, 0.99)
    assert abs(float(lam) - 0.91) < 1e-6
    lam = O.anb_step(np.float32(0.9), False, 0.01, 0.8, 0.99)
    assert abs(float(lam) - 0.89) < 1e-6
    om, tau = O.tam_threshold(np.float32(0.95), np.float32(0.01))
    assert abs(float(om) - 0.05) < 1e-7 and abs(float(tau) - 0.06) < 1e-7


def test_tam_candidate_is_strict():
    """The page asks for scores that EXCEED tau: a score equal to tau is not a
    candidate, the next float32 above it is."""
    om, tau = O.tam_threshold(LAM, EPS)
    s = np.array([tau, np.nextafter(tau, np.float32(np.inf)), np.nextafter(tau, np.float32(0))],
                 dtype=np.float32)
    cand, topk = O.tam_select(s, tau, 5)
    assert cand.tolist() == [False, True, False] and topk.tolist() == [1]


# ---------------------------------------------------------------- 8-bit quantized rows

def test_q8_hand_computed():
    """One neuron, d = 4: u = 0.5 * (q_up . x), ReLU, y = h * 0.25 * q_down."""
    up_q = np.array([[1, -2, 3, 0]], dtype=np.int8)
    x = np.array([1.0, 2.0, -1.0, 3.0])                        # q . x = 1 - 4 - 3 + 0 = -6
    x2 = np.array([2.0, 0.0, 1.0, 1.0])                        # q . x2 = 2 + 0 + 3 + 0 = 5
    down_q = np.array([[2], [0], [-1], [4]], dtype=np.int8)
    s_up = np.array([0.5], dtype=np.float32)
    s_dn = np.array([0.25], dtype=np.float32)
    y, h = O.ffn_sparse_q8(x2, up_q, s_up, None, None, down_q, s_dn, "relu", np.array([True]))
    assert h.tolist() == [2.5]                                 # 0.5 * 5
    assert y.tolist() == [1.25, 0.0, -0.625, 2.5]              # 2.5 * 0.25 * [2, 0, -1, 4]
    y0, _ = O.ffn_sparse_q8(x, up_q, s_up, None, None, down_q, s_dn, "relu", np.array([True]))
    assert (y0 == 0.0).all()                                   # u = -3 < 0


@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu", "relu2"])
def test_q8_all_active_equals_library_dense(act):
    """Codes times per-neuron scales, dequantized by torch and run through a
    library dense FFN, equal the oracle's quantized sparse FFN with every
    neuron active (scales differ per neuron, so a scale applied along the
    wrong axis fails)."""
    rng = np.random.default_rng(11)
    d, f = 24, 64
    up_q = rng.integers(-127, 128, (f, d)).astype(np.int8)
    gate_q = rng.integers(-127, 128, (f, d)).astype(np.int8) if act in ("reglu", "swiglu") else None
    down_q = rng.integers(-127, 128, (d, f)).astype(np.int8)
    s_up = rng.uniform(1e-3, 2e-2, f).astype(np.float32)
    s_g = rng.uniform(1e-3, 2e-2, f).astype(np.float32)
    s_dn = rng.uniform(1e-3, 2e-2, f).astype(np.float32)
    perm = rng.permutation(f)
    x = rng.standard_normal(d)
    y, _ = O.ffn_sparse_q8(x, up_q, s_up, gate_q, s_g if gate_q is not None else None, down_q, s_dn, act,
                           np.ones(f, dtype=bool), perm)
    up = torch.from_numpy(up_q).double() * torch.from_numpy(s_up).double()[:, None]
    gate = (torch.from_numpy(gate_q).double() * torch.from_numpy(s_g).double()[:, None]).numpy() \
        if gate_q is not None else None
    down = torch.from_numpy(down_q).double() * torch.from_numpy(s_dn).double()[None, :]
    ref = _torch_dense(x, up.numpy(), gate, down.numpy(), act)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_q4_storage_hand_computed():
    """Codes 1, -2 -> low half 0x1, high half (-2 mod 16) = 0xE: byte 0xE1;
    -8, 7 -> 0x8 | 0x70 = 0x78; 0, -1 -> 0xF0."""
    b = O.pack_q4(np.array([1, -2, -8, 7, 0, -1], dtype=np.int8))
    assert b.tolist() == [0xE1, 0x78, 0xF0]
    assert O.unpack_q4(b).tolist() == [1, -2, -8, 7, 0, -1]


def test_q4_storage_roundtrip_every_pair():
    c = np.array([[a, b] for a in range(-8, 8) for b in range(-8, 8)], dtype=np.int8)
    packed = O.pack_q4(c)
    assert packed.shape == (256, 1) and sorted(packed[:, 0].tolist()) == list(range(256))
    assert (O.unpack_q4(packed) == c).all()


def test_q4_range_and_arithmetic():
    """4-bit rows use the 8-bit arithmetic (code x scale); codes outside
    [-8, 7] are refused."""
    rng = np.random.default_rng(5)
    d, f = 16, 32
    up_q = rng.integers(-8, 8, (f, d)).astype(np.int8)
    down_q = rng.integers(-8, 8, (d, f)).astype(np.int8)
    s_up = rng.uniform(1e-2, 1e-1, f).astype(np.float32)
    s_dn = rng.uniform(1e-2, 1e-1, f).astype(np.float32)
    x = rng.standard_normal(d)
    act = rng.random(f) < 0.5
    y4, h4 = O.ffn_sparse_q4(x, up_q, s_up, None, None, down_q, s_dn, "relu", act)
    U = up_q.astype(np.float64) * s_up.astype(np.float64)[:, None]
    D = down_q.astype(np.float64) * s_dn.astype(np.float64)[None, :]
    h = np.maximum(U[act] @ x, 0.0)
    assert np.allclose(y4, D[:, act] @ h, rtol=1e-13, atol=1e-13) and np.allclose(h4, h, rtol=1e-13, atol=0)
    bad = up_q.copy()
    bad[0, 0] = 8
    with pytest.raises(ValueError):
        O.ffn_sparse_q4(x, bad, s_up, None, None, down_q, s_dn, "relu", act)


# ---------------------------------------------------------------- stored weights and the dense form

def _store(w, dtype):
    """Round float64 weights to the stored type with torch (round to nearest
    even) and return (stored array as the oracle takes it, torch's own widened
    float64 values of the stored weights)."""
    t = torch.from_numpy(w)
    if dtype == "f32":
        s = t.float()
        return s.numpy(), s.double().numpy()
    if dtype == "f16":
        s = t.half()
        return s.numpy(), s.double().numpy()
    s = t.to(torch.bfloat16)
    return s.view(torch.int16).numpy().view(np.uint16), s.double().numpy()


@pytest.mark.parametrize("dtype,act", [("f32", "relu"), ("f16", "swiglu"), ("bf16", "reglu"), ("bf16", "relu2")])
def test_stored_weights_equal_library_on_torch_widened_values(dtype, act):
    """The stored-weight form reads only active rows and columns, widens them
    and applies the definition; it must equal a library dense FFN on torch's
    own widening of the same stored weights, with the inactive neurons zeroed
    through the neuron table."""
    rng = np.random.default_rng(21)
    d, f = 16, 64
    up, gate, down = _rand_layer(rng, d, f, act)
    up_s, up_w = _store(up, dtype)
    gate_s, gate_w = _store(gate, dtype) if gate is not None else (None, None)
    down_s, down_w = _store(down, dtype)
    perm = rng.permutation(f)
    for trial in range(20):
        x = rng.standard_normal(d)
        act_slots = rng.random(f) < 0.3
        y, _ = O.ffn_sparse_stored(x, up_s, gate_s, down_s, dtype, act, act_slots, perm)
        keep = np.zeros(f, dtype=bool)
        keep[perm[act_slots]] = True
        ref = _torch_dense(x, up_w * keep[:, None], gate_w * keep[:, None] if gate_w is not None else None,
                           down_w * keep[None, :], act)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12), trial


@pytest.mark.parametrize("act", ["relu", "reglu", "swiglu", "relu2"])
def test_dense_form_equals_library(act):
    rng = np.random.default_rng(22)
    up, gate, down = _rand_layer(rng, 24, 64, act)
    x = rng.standard_normal(24)
    assert np.allclose(O.ffn_dense(x, up, gate, down, act), _torch_dense(x, up, gate, down, act),
                       rtol=1e-12, atol=1e-12)
