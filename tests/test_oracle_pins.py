"""Pins of the float64 oracle to facts outside itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, an
inverted or missing scale, a transposed operand, a wrong adapter index, an
off-by-one loop bound) fails at least one of them; ``test_mutations_fail_pins``
plants those slips in a copy of the C source and checks exactly that.

Pins:
  * hand-worked dyadic cases (tests/golden/hand_worked.json), exact;
  * the folded form (W + (alpha/r) B A) x in exact rational arithmetic on
    tiny integer inputs, with non-dyadic scales ("Your LoRA Adapters Are
    Thrashing Your GPUs", §02 "Weight merging vs. keeping adapters separate":
    merged and additive serving give the same layer);
  * the folded form in float64 through numpy matmul on a mixed-rank case;
  * base-only rows equal the plain library product x W^T;
  * row permutation permutes the outputs bit for bit (rows are independent);
  * a numpy restatement of the adapted_linear sketch ("Adapter Residency…",
    §"What the forward pass has to do differently"), looping over adapters
    instead of over rows.
"""

import json
import os
import shutil
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import make_config, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _case_inputs(case):
    x = np.asarray(case["x"], np.float32)
    W = np.asarray(case["W"], np.float32)
    ids = np.asarray(case["row_adapter"], np.int32)
    ranks = np.asarray([a["r"] for a in case["adapters"]], np.int32)
    alphas = np.asarray([a["alpha"] for a in case["adapters"]], np.float64)
    adapters = {i: (np.asarray(a["A"], np.float32), np.asarray(a["B"], np.float32))
                for i, a in enumerate(case["adapters"])}
    return x, W, ids, ranks, alphas, adapters


# --------------------------------------------------------------------------
# pin functions: return a list of failure descriptions (empty = pass)
# --------------------------------------------------------------------------

def pin_hand_worked(lib=None):
    fails = []
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        x, W, ids, ranks, alphas, adapters = _case_inputs(case)
        y = oracle.forward(x, W, ids, ranks, alphas, adapters, threads=2, lib=lib)
        want = np.asarray(case["y"], np.float64)
        if not np.array_equal(y, want):
            fails.append(f"{case['name']}: got {y.tolist()} want {want.tolist()}")
    return fails


def _rational_case(seed):
    rng = np.random.default_rng(seed)
    M, K, N = 6, 5, 4
    ranks = np.array([1, 2, 3], np.int32)
    alphas = np.array([1.0, 3.0, 5.0])  # scales 1, 3/2, 5/3
    x = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    W = rng.integers(-3, 4, size=(N, K)).astype(np.float32)
    adapters = {i: (rng.integers(-3, 4, size=(int(r), K)).astype(np.float32),
                    rng.integers(-3, 4, size=(N, int(r))).astype(np.float32))
                for i, r in enumerate(ranks)}
    ids = np.array([0, 1, 2, -1, 2, 1], np.int32)
    return x, W, ids, ranks, alphas, adapters


def _folded_exact(x, W, ids, ranks, alphas, adapters):
    """y = (W + s B A) x with the merged matrix built first, in exact rationals."""
    M, K = x.shape
    N = W.shape[0]
    out = []
    for m in range(M):
        i = int(ids[m])
        Wm = [[Fraction(int(W[n, k])) for k in range(K)] for n in range(N)]
        if i >= 0:
            A, B = adapters[i]
            s = Fraction(int(alphas[i])) / Fraction(int(ranks[i]))
            for n in range(N):
                for k in range(K):
                    Wm[n][k] += s * sum(Fraction(int(B[n, j])) * Fraction(int(A[j, k]))
                                        for j in range(int(ranks[i])))
        out.append([sum(Wm[n][k] * Fraction(int(x[m, k])) for k in range(K)) for n in range(N)])
    return out


def pin_folded_rational(lib=None):
    fails = []
    for seed in (3, 4):
        args = _rational_case(seed)
        y = oracle.forward(*args, threads=2, lib=lib)
        exact = _folded_exact(*args)
        for m, row in enumerate(exact):
            bound = 1e-12 * (max(abs(float(v)) for v in row) + 1.0)
            for n, v in enumerate(row):
                if abs(y[m, n] - float(v)) > bound:
                    fails.append(f"seed {seed} row {m} col {n}: {y[m, n]} vs {v}")
    return fails


def _mixed_case():
    return synth("pin_mixed", M=40, K=96, Ns=[80], num_slots=5,
                 rank_choices=(1, 3, 8, 16), dtype="bf16", seed=7, none_frac=0.2)


def pin_folded_float64(lib=None):
    wl = _mixed_case()
    W = wl.projections[0].W.astype(np.float64)
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    y = oracle.forward(wl.x, wl.projections[0].W, wl.row_adapter, wl.ranks, wl.alphas,
                       adapters, threads=2, lib=lib)
    fails = []
    for m in range(wl.M):
        i = int(wl.row_adapter[m])
        Wm = W.copy()
        if i >= 0:
            A, B = adapters[i]
            Wm += (float(wl.alphas[i]) / float(wl.ranks[i])) * (B.astype(np.float64) @ A.astype(np.float64))
        ref = Wm @ wl.x[m].astype(np.float64)
        err = np.max(np.abs(y[m] - ref))
        if err > 1e-12 * (np.max(np.abs(ref)) + 1.0):
            fails.append(f"row {m}: max err {err}")
    return fails


def pin_base_rows(lib=None):
    wl = _mixed_case()
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    y = oracle.forward(wl.x, wl.projections[0].W, wl.row_adapter, wl.ranks, wl.alphas,
                       adapters, threads=2, lib=lib)
    ref = wl.x.astype(np.float64) @ wl.projections[0].W.astype(np.float64).T
    fails = []
    base = np.nonzero(wl.row_adapter < 0)[0]
    assert base.size > 0
    for m in base:
        err = np.max(np.abs(y[m] - ref[m]))
        if err > 1e-12 * (np.max(np.abs(ref[m])) + 1.0):
            fails.append(f"base row {m}: max err {err}")
    return fails


ALL_PINS = [pin_hand_worked, pin_folded_rational, pin_folded_float64, pin_base_rows]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    assert pin() == []


def test_base_only_rows_bit_identical_without_adapters():
    """A row with id -1 gives the very bits of the adapter-free evaluation."""
    wl = _mixed_case()
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    W = wl.projections[0].W
    y = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters, threads=3)
    y0 = oracle.forward(wl.x, W, np.full(wl.M, -1, np.int32), wl.ranks, wl.alphas, {}, threads=1)
    base = wl.row_adapter < 0
    assert np.array_equal(y[base], y0[base])
    # and every adapted row differs from its base-only value
    assert np.all(np.max(np.abs(y[~base] - y0[~base]), axis=1) > 0)


def test_permutation_equivariance_bitwise():
    wl = _mixed_case()
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    W = wl.projections[0].W
    y = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters, threads=4)
    perm = np.random.default_rng(11).permutation(wl.M)
    yp = oracle.forward(wl.x[perm], W, wl.row_adapter[perm], wl.ranks, wl.alphas, adapters, threads=1)
    assert np.array_equal(yp, y[perm])


def test_row_subset_matches_full():
    wl = _mixed_case()
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    W = wl.projections[0].W
    y = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters)
    rows = [39, 0, 17, 17, 5]
    ys = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters, rows=rows)
    assert np.array_equal(ys, y[rows])


def test_scale_is_linear_in_alpha():
    """Doubling every alpha doubles each row's correction (the scale enters
    once, multiplying B (A x))."""
    wl = _mixed_case()
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    W = wl.projections[0].W
    none = np.full(wl.M, -1, np.int32)
    y0 = oracle.forward(wl.x, W, none, wl.ranks, wl.alphas, {})
    y1 = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters)
    y2 = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, 2 * wl.alphas.astype(np.float64), adapters)
    d1, d2 = y1 - y0, y2 - y0
    assert np.allclose(d2, 2 * d1, rtol=1e-12, atol=1e-12)


def test_sgmv_segments_equal_bgmv_ids():
    """The same assignment given as sorted segments + permutation or as
    per-row ids gives bit-identical outputs."""
    wl = _mixed_case()
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    W = wl.projections[0].W
    perm, offs, seg_adapter = oracle.segment_rows(wl.row_adapter, wl.num_slots)
    ids = oracle.rows_from_segments(wl.M, offs, seg_adapter, perm)
    assert np.array_equal(ids, wl.row_adapter)
    y = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters)
    ys = oracle.forward(wl.x, W, ids, wl.ranks, wl.alphas, adapters)
    assert np.array_equal(y, ys)


def _adapted_linear_numpy(x, W, ids, ranks, alphas, adapters):
    """Loop over adapters (not rows): dense base, then for each adapter the
    gathered rows go through the rank-r bottleneck and are added back with
    the adapter's scale."""
    x64 = x.astype(np.float64)
    out = x64 @ W.astype(np.float64).T
    for i, (A, B) in adapters.items():
        rows = np.nonzero(ids == i)[0]
        if rows.size == 0:
            continue
        low = (x64[rows] @ A.astype(np.float64).T) @ B.astype(np.float64).T
        out[rows] += (float(alphas[i]) / float(ranks[i])) * low
    return out


@pytest.mark.parametrize("cfg", ["tiny_fp32", "decode_bgmv"])
def test_numpy_restatement_agrees(cfg):
    wl = make_config(cfg)
    adapters = {i: wl.adapter(0, i) for i in wl.used_slots}
    W = wl.projections[0].W
    y = oracle.forward(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters)
    ref = _adapted_linear_numpy(wl.x, W, wl.row_adapter, wl.ranks, wl.alphas, adapters)
    scale = np.max(np.abs(ref), axis=1, keepdims=True) + 1.0
    assert np.max(np.abs(y - ref) / scale) < 1e-12


def test_oracle_rejects_bad_ids():
    x, W, ids, ranks, alphas, adapters = _case_inputs(json.load(open(GOLDEN))["cases"][1])
    bad = ids.copy()
    bad[0] = 7
    with pytest.raises(ValueError):
        oracle.forward(x, W, bad, ranks, alphas, adapters)
    with pytest.raises(ValueError):
        oracle.forward(x, W, ids, ranks, alphas, {0: adapters[0]})


# --------------------------------------------------------------------------
# planted mistakes: every one must fail at least one pin
# --------------------------------------------------------------------------

MUTATIONS = {
    "drop_scale": ("yr[n] += s * t;", "yr[n] += t;"),
    "inverse_scale": ("const double s = J->alphas[i] / (double)r;",
                      "const double s = (double)r / J->alphas[i];"),
    "wrong_sign": ("yr[n] += s * t;", "yr[n] -= s * t;"),
    "B_transposed": ("t += (double)br[j] * v_scratch[j];",
                     "t += (double)Bi[(size_t)j * (size_t)J->N + (size_t)n] * v_scratch[j];"),
    "A_transposed": ("t += (double)ar[k] * (double)xr[k];",
                     "t += (double)Ai[(size_t)k * (size_t)r + (size_t)j] * (double)xr[k];"),
    "W_transposed": ("acc += (double)wr[k] * (double)xr[k];",
                     "acc += (double)J->W[(size_t)k * (size_t)J->N + (size_t)n] * (double)xr[k];"),
    "drop_base": ("yr[n] = acc;", "yr[n] = 0.0;"),
    "next_adapter": ("const int i = J->row_adapter[m];",
                     "const int i = (J->row_adapter[m] < 0) ? -1 : (J->row_adapter[m] + 1) % J->num_adapters;"),
    "base_k_off_by_one": ("for (int k = 0; k < J->K; ++k)\n            acc +=",
                          "for (int k = 1; k < J->K; ++k)\n            acc +="),
    "expand_rank_off_by_one": ("for (int j = 0; j < r; ++j)\n            t += (double)br[j]",
                               "for (int j = 1; j < r; ++j)\n            t += (double)br[j]"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_mutations_fail_pins():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")).read()
    tmp = tempfile.mkdtemp(prefix="oracle_mut_")
    try:
        for name, (old, new) in MUTATIONS.items():
            assert src.count(old) == 1, f"mutation {name}: pattern not found once"
            path_c = os.path.join(tmp, f"{name}.c")
            path_so = os.path.join(tmp, f"{name}.so")
            with open(path_c, "w") as f:
                f.write(src.replace(old, new))
            subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                            path_c, "-o", path_so], check=True)
            lib = oracle.load_library(path_so)
            caught = [p.__name__ for p in ALL_PINS if p(lib=lib)]
            assert caught, f"planted mistake '{name}' passed every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
