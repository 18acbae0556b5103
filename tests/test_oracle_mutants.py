"""Planted mistakes in the CPU oracle, each of which the pins must catch.

The oracle is trusted only because its pins (tests/test_oracle_pins.py) tie
it to facts that do not come from the oracle itself. This file checks that
claim the other way round: it swaps one oracle function at a time for a copy
with one plausible mistake in it (a dropped ReLU or bias, a wrong sign, a
transposed or mis-indexed operand, a non-strict comparison, a swapped set, a
wrong bit or half-byte order) and runs the pins named for that mistake. Each
of them must fail. A control run checks that the same runner passes every pin
on the unchanged oracle. Everything runs on the CPU; the mistakes live only
in this process, inside the patched oracle module.
"""

import inspect
import itertools
import json
import os
import warnings

import numpy as np
import pytest

import test_oracle_pins as P
from oracle import sffn_oracle as O

with open(os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")) as _fh:
    _GOLDEN = json.load(_fh)

_ORIG = {n: getattr(O, n) for n in dir(O) if callable(getattr(O, n)) and not n.startswith("_")}


def _pin_cases():
    """Every pin function with each of its parametrize combinations."""
    for name, fn in sorted(vars(P).items()):
        if not (name.startswith("test_") and inspect.isfunction(fn)):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = mark.args[0]
            names = [s.strip() for s in names.split(",")] if isinstance(names, str) else list(names)
            grids.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in mark.args[1]])
        for combo in (itertools.product(*grids) if grids else [()]):
            kw = {}
            for part in combo:
                kw.update(part)
            if "golden" in inspect.signature(fn).parameters:
                kw["golden"] = _GOLDEN
            yield name, fn, kw


def _fails(fn, kw) -> bool:
    try:
        with warnings.catch_warnings(), np.errstate(all="ignore"):
            warnings.simplefilter("ignore")
            fn(**kw)
    except (Exception, pytest.fail.Exception):
        return True
    return False


def _failing(names=None):
    """Names of the pins (of those listed, else all) that fail; a pin with
    several parameter sets fails if any of them fails."""
    out = set()
    for name, fn, kw in _pin_cases():
        if (names is None or name in names) and name not in out and _fails(fn, kw):
            out.add(name)
    return out


# ----------------------------------------------------------------- the planted mistakes

def _hidden_without_relu(W1, x, b1=None):
    pre = W1 @ x
    return pre if b1 is None else pre + b1


def _hidden_bias_after_relu(W1, x, b1=None):
    hid = np.maximum(W1 @ x, 0.0)
    return hid if b1 is None else hid + b1


def _scores_without_bias(W2, hid, b2=None):
    return W2 @ hid


def _threshold_strict(scores, thres):
    return np.asarray(scores > thres, dtype=bool)


def _threshold_nan_active(scores, thres):
    return ~np.asarray(scores < thres, dtype=bool)


def _words_msb_first(bits):
    words = np.zeros((bits.shape[0] + 31) // 32, dtype=np.uint32)
    for i in np.flatnonzero(bits):
        words[i // 32] |= np.uint32(1) << np.uint32(31 - i % 32)
    return words


def _group_all_members(active, group_size):
    return active.reshape(-1, group_size).all(axis=1)


def _group_strided(active, group_size):
    return active.reshape(group_size, -1).any(axis=0)


def _views_descending(active, group_size):
    v = _ORIG["mask_views"](active, group_size)
    v["idx"] = v["idx"][::-1].copy()
    return v


def _act_with(**swap):
    def act(a, u, g):
        if a in swap:
            return swap[a](u, g)
        return _ORIG["activation"](a, u, g)
    return act


def _ffn_down_by_slot(x, up, gate, down, act, active, perm=None):
    perm = np.arange(up.shape[0]) if perm is None else np.asarray(perm)
    slots = np.flatnonzero(active)
    orig = perm[slots]
    g = gate[orig] @ x if gate is not None else None
    h = O.activation(act, up[orig] @ x, g)
    return down[:, slots] @ h, h


def _ffn_up_by_slot(x, up, gate, down, act, active, perm=None):
    perm = np.arange(up.shape[0]) if perm is None else np.asarray(perm)
    slots = np.flatnonzero(active)
    orig = perm[slots]
    g = gate[slots] @ x if gate is not None else None
    h = O.activation(act, up[slots] @ x, g)
    return down[:, orig] @ h, h


def _ffn_ignores_mask(x, up, gate, down, act, active, perm=None):
    return _ORIG["ffn_sparse"](x, up, gate, down, act, np.ones(up.shape[0], dtype=bool), None)


def _zero_skip_counts_every_active(x, up, gate, down, act, active, perm=None):
    y, _ = _ORIG["ffn_sparse_zero_skip"](x, up, gate, down, act, active, perm)
    return y, int(np.count_nonzero(active))


def _zero_skip_drops_negative(x, up, gate, down, act, active, perm=None):
    perm = np.arange(up.shape[0]) if perm is None else np.asarray(perm)
    orig = perm[np.flatnonzero(active)]
    g = gate[orig] @ x if gate is not None else None
    h = O.activation(act, up[orig] @ x, g)
    keep = h > 0.0
    return down[:, orig[keep]] @ h[keep], int(keep.sum())


def _stored_ignores_perm(x, up_s, gate_s, down_s, dtype, act, active, perm=None):
    return _ORIG["ffn_sparse_stored"](x, up_s, gate_s, down_s, dtype, act, active, None)


def _q8_down_scaled_by_up(x, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, act, active, perm=None):
    return _ORIG["ffn_sparse_q8"](x, up_q, up_scale, gate_q, gate_scale, down_q, up_scale, act, active, perm)


def _q8_down_scale_per_output(x, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, act, active, perm=None):
    f = up_q.shape[0]
    perm = np.arange(f) if perm is None else np.asarray(perm)
    orig = perm[np.flatnonzero(active)]
    U = up_q[orig].astype(np.float64) * up_scale[orig].astype(np.float64)[:, None]
    G = None if gate_q is None else gate_q[orig].astype(np.float64) * gate_scale[orig].astype(np.float64)[:, None]
    D = down_q[:, orig].astype(np.float64) * down_scale[:down_q.shape[0]].astype(np.float64)[:, None]
    return O.ffn_sparse(x, U, G, D, act, np.ones(orig.shape[0], dtype=bool), None)


def _pack_q4_high_first(codes):
    c = np.asarray(codes).astype(np.int16)
    return ((c[..., 1::2] & 15) | ((c[..., 0::2] & 15) << 4)).astype(np.uint8)


def _unpack_q4_unsigned(packed):
    b = np.asarray(packed).astype(np.int16)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int16)
    out[..., 0::2], out[..., 1::2] = b & 15, b >> 4
    return out.astype(np.int8)


def _widen_bf16_as_f16(a, dtype):
    if dtype == "bf16":
        return np.asarray(a, dtype=np.uint16).view(np.float16).astype(np.float64)
    return _ORIG["widen"](a, dtype)


def _tam_adds_one(scores, gactive, lam, eps):
    lam = np.float32(lam)
    _, tau = O.tam_threshold(lam, eps)
    s = (lam * np.asarray(scores, dtype=np.float32)).astype(np.float32)
    return (s + np.where(gactive, np.float32(1), np.float32(0))).astype(np.float32), tau


def _tam_decays_only_when_idle(scores, gactive, lam, eps):
    lam = np.float32(lam)
    om, tau = O.tam_threshold(lam, eps)
    s = np.asarray(scores, dtype=np.float32)
    return np.where(gactive, (s + om).astype(np.float32), (lam * s).astype(np.float32)), tau


def _tau_without_eps(lam, eps):
    om = np.float32(np.float32(1.0) - np.float32(lam))
    return om, om


def _select_non_strict(scores, tau, capacity_k):
    s = np.asarray(scores, dtype=np.float32)
    cand = s >= np.float32(tau)
    ids = np.flatnonzero(cand)
    order = ids[np.argsort(-s[ids].astype(np.float64), kind="stable")]
    return cand, order[:max(0, min(int(capacity_k), order.shape[0]))].astype(np.int32)


def _select_ties_to_higher_index(scores, tau, capacity_k):
    s = np.asarray(scores, dtype=np.float32)
    cand = s > np.float32(tau)
    ids = np.flatnonzero(cand)[::-1]
    order = ids[np.argsort(-s[ids].astype(np.float64), kind="stable")]
    return cand, order[:max(0, min(int(capacity_k), order.shape[0]))].astype(np.int32)


def _update_swaps_load_evict(scores, prev_resident, gactive, lam, eps, capacity_k):
    r = _ORIG["tam_update"](scores, prev_resident, gactive, lam, eps, capacity_k)
    r["load"], r["evict"] = r["evict"], r["load"]
    return r


def _anb_reversed(lam, stall_io, alpha, lo, hi):
    return _ORIG["anb_step"](lam, not stall_io, alpha, lo, hi)


def _union_is_intersection(actives, group_size):
    v = O.mask_views(np.asarray(actives, dtype=bool).all(axis=0), group_size)
    return {"active": np.asarray(actives, dtype=bool).all(axis=0), "unmask": v["nmask"], "ugmask": v["gmask"],
            "uidx": v["idx"], "ucount": v["count"]}


def _decode_scores_unpermuted(x, W1, W2, up, gate, down, act, thres, group_size, perm=None, b1=None, b2=None,
                              active_override=None):
    f = W2.shape[0]
    perm = np.arange(f) if perm is None else np.asarray(perm)
    scores = O.predictor_scores(W2, O.predictor_hidden(W1, x, b1), b2)      # left in original order
    active = O.active_from_scores(scores, thres)
    views = O.mask_views(active, group_size)
    y, h = O.ffn_sparse(x, up, gate, down, act, active, perm)
    return {"scores": scores, "active": active, "y": y, "h": h, **views}


def _closed_form_extra_power(acts, lam, s0=0.0):
    a = np.asarray(acts, dtype=np.float64)
    T = a.shape[0]
    return float(lam ** T * s0 + (1.0 - lam) * sum(lam ** (T - t + 1) * a[t - 1] for t in range(1, T + 1)))


def _dense_without_activation(x, up, gate, down, act):
    return down @ (up @ x)


# (oracle function, its mistaken copy, the pins that must catch it)
MUTANTS = {
    "hidden layer without its ReLU": ("predictor_hidden", _hidden_without_relu,
                                      ["test_predictor_closed_form", "test_all_active_equals_library_dense"]),
    "hidden bias added after the ReLU": ("predictor_hidden", _hidden_bias_after_relu,
                                         ["test_predictor_biases_shift_scores"]),
    "output bias dropped": ("predictor_scores", _scores_without_bias,
                            ["test_predictor_biases_shift_scores", "test_brute_force_scalar_predictor_d8"]),
    "threshold test > instead of >=": ("active_from_scores", _threshold_strict,
                                       ["test_predictor_closed_form", "test_threshold_nan_and_equality"]),
    "NaN score counted active": ("active_from_scores", _threshold_nan_active,
                                 ["test_threshold_nan_and_equality"]),
    "bits stored most significant first": ("bits_to_words", _words_msb_first,
                                           ["test_bit_layout_roundtrip", "test_predictor_closed_form",
                                            "test_group_mask_size_64"]),
    "group active only when all members are": ("group_active", _group_all_members,
                                               ["test_group_mask_size_64", "test_predictor_closed_form",
                                                "test_batch_union_and_identical_tokens"]),
    "groups taken as strided, not contiguous, slots": ("group_active", _group_strided,
                                                       ["test_group_mask_size_64"]),
    "index list in descending order": ("mask_views", _views_descending, ["test_predictor_closed_form"]),
    "ReGLU gates the wrong operand": ("activation", _act_with(reglu=lambda u, g: np.maximum(u, 0.0) * g),
                                      ["test_ffn_reglu_closed_form", "test_ffn_swiglu_relu_closed_form",
                                       "test_all_active_equals_library_dense"]),
    "SiLU with the sign of the exponent flipped": (
        "activation", _act_with(swiglu=lambda u, g: g / (1.0 + np.exp(g)) * u),
        ["test_ffn_swiglu_relu_closed_form", "test_all_active_equals_library_dense"]),
    "SiLU without its factor g (sigmoid gate)": (
        "activation", _act_with(swiglu=lambda u, g: u / (1.0 + np.exp(-g))),
        ["test_ffn_swiglu_relu_closed_form", "test_all_active_equals_library_dense"]),
    "squared ReLU not squared": ("activation", _act_with(relu2=lambda u, g: np.maximum(u, 0.0)),
                                 ["test_ffn_swiglu_relu_closed_form", "test_all_active_equals_library_dense"]),
    "down columns indexed by slot, not neuron": ("ffn_sparse", _ffn_down_by_slot,
                                                 ["test_all_active_equals_library_dense",
                                                  "test_brute_force_masks_d8", "test_permutation_invariance"]),
    "up/gate rows indexed by slot, not neuron": ("ffn_sparse", _ffn_up_by_slot,
                                                 ["test_all_active_equals_library_dense",
                                                  "test_brute_force_masks_d8"]),
    "mask ignored (dense FFN)": ("ffn_sparse", _ffn_ignores_mask,
                                 ["test_ffn_reglu_closed_form", "test_none_active_is_exact_zero",
                                  "test_brute_force_masks_d8"]),
    "zero-skip counts every active column": ("ffn_sparse_zero_skip", _zero_skip_counts_every_active,
                                             ["test_zero_skip_hand_computed",
                                              "test_zero_skip_equals_full_and_library"]),
    "zero-skip drops negative activations": ("ffn_sparse_zero_skip", _zero_skip_drops_negative,
                                             ["test_zero_skip_hand_computed",
                                              "test_zero_skip_equals_full_and_library"]),
    "stored-weight form ignores the neuron table": ("ffn_sparse_stored", _stored_ignores_perm,
                                                    ["test_stored_weights_equal_library_on_torch_widened_values"]),
    "down codes scaled by the up scales": ("ffn_sparse_q8", _q8_down_scaled_by_up,
                                           ["test_q8_hand_computed", "test_q8_all_active_equals_library_dense"]),
    "down scale applied per output, not per neuron": ("ffn_sparse_q8", _q8_down_scale_per_output,
                                                      ["test_q8_all_active_equals_library_dense"]),
    "4-bit codes stored high half first": ("pack_q4", _pack_q4_high_first, ["test_q4_storage_hand_computed"]),
    "4-bit codes read without sign": ("unpack_q4", _unpack_q4_unsigned,
                                      ["test_q4_storage_hand_computed", "test_q4_storage_roundtrip_every_pair"]),
    "bfloat16 read as float16": ("widen", _widen_bf16_as_f16,
                                 ["test_widen_exact", "test_stored_weights_equal_library_on_torch_widened_values"]),
    "momentum adds 1, not 1 - lambda": ("tam_scores_step", _tam_adds_one,
                                        ["test_tam_isolated_hit_never_candidate",
                                         "test_tam_matches_closed_form_random_sequences"]),
    "momentum decays only on idle steps": ("tam_scores_step", _tam_decays_only_when_idle,
                                           ["test_tam_two_hits_and_gap_rule",
                                            "test_tam_matches_closed_form_random_sequences"]),
    "tau without eps": ("tam_threshold", _tau_without_eps,
                        ["test_tam_two_hits_and_gap_rule", "test_anb_step_clamps_and_moves"]),
    "candidate test >= tau": ("tam_select", _select_non_strict, ["test_tam_candidate_is_strict"]),
    "top-K ties to the higher group index": ("tam_select", _select_ties_to_higher_index,
                                             ["test_tam_topk_against_rank_definition"]),
    "load and evict sets swapped": ("tam_update", _update_swaps_load_evict, ["test_tam_update_sets"]),
    "balancer moves lambda the wrong way": ("anb_step", _anb_reversed, ["test_anb_step_clamps_and_moves"]),
    "batch union taken as intersection": ("batch_union", _union_is_intersection,
                                          ["test_batch_union_and_identical_tokens"]),
    "scores left in neuron order, not slot order": ("decode_layer", _decode_scores_unpermuted,
                                                    ["test_all_active_equals_library_dense",
                                                     "test_brute_force_scalar_predictor_d8",
                                                     "test_permutation_invariance"]),
    "closed form with one power of lambda too many": ("tam_closed_form", _closed_form_extra_power,
                                                      ["test_tam_matches_closed_form_random_sequences"]),
    "dense form without the activation": ("ffn_dense", _dense_without_activation,
                                          ["test_dense_form_equals_library"]),
}


def test_runner_passes_every_pin_on_the_unchanged_oracle():
    cases = list(_pin_cases())
    assert len({name for name, _, _ in cases}) >= 30
    assert _failing() == set()


@pytest.mark.parametrize("mistake", sorted(MUTANTS))
def test_planted_mistake_is_caught(mistake, monkeypatch):
    target, mutant, catchers = MUTANTS[mistake]
    assert target in _ORIG and all(c in vars(P) for c in catchers)
    monkeypatch.setattr(O, target, mutant)
    failed = _failing(set(catchers))
    assert failed == set(catchers), f"{mistake}: not caught by {sorted(set(catchers) - failed)}"
