"""Pins for the fp64 oracle: it is checked against what the pages and the
mathematics fix, never against itself or the CUDA path.

Each pin is a function of an implementation ``ref(q, k, v, causal, scale) ->
(O, LSE)`` on float64 [B, S, H, D] arrays, so that ``test_pins_catch_planted_
mistakes`` can run the same pins on deliberately broken copies of the oracle
(planted on the CPU) and show that each plausible mistake fails at least one.
"""
import math
import os

import numpy as np
import pytest

import fa_inputs
from oracle import (attention_reference, attention_reference_f64, attention_reference_varlen,
                    attention_rows, decode_bf16, decode_f16,
                    online_softmax_attention, softmax_probabilities)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _parse_golden(name):
    env = {"ln": math.log}
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            vals = [float(eval(tok, {"__builtins__": {}}, env))
                    for tok in val.split()]
            out[key] = vals if len(vals) > 1 else vals[0]
    return out


# ---------------------------------------------------------------------------
# pins (each takes an implementation)

def pin_golden_worked_example(ref):
    g = _parse_golden("worked_example_two_tiles.txt")
    q = np.array(g["q"]).reshape(1, 4, 1, 1)
    k = np.array(g["k"]).reshape(1, 4, 1, 1)
    v = np.array(g["v"]).reshape(1, 4, 1, 1)
    O, L = ref(q, k, v, False, g["scale"])
    np.testing.assert_allclose(O[0, :, 0, 0], g["noncausal_O"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(L[0, 0, :], g["noncausal_LSE"], rtol=0, atol=1e-13)
    O, L = ref(q, k, v, True, g["scale"])
    np.testing.assert_allclose(O[0, :, 0, 0], g["causal_O"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(L[0, 0, :], g["causal_LSE"], rtol=0, atol=1e-13)


def pin_uniform_scores(ref):
    g = _parse_golden("uniform_scores_n320.txt")
    S = int(g["S"])
    q = np.zeros((1, S, 1, 2))
    k = np.stack([np.arange(S) % 7, -np.ones(S)], axis=1).reshape(1, S, 1, 2)
    v = np.stack([np.arange(S), np.ones(S)], axis=1).reshape(1, S, 1, 2).astype(float)
    O, L = ref(q, k, v, False, g["scale"])
    np.testing.assert_allclose(O[0, :, 0, 0], g["noncausal_O0"], atol=1e-10)
    np.testing.assert_allclose(O[0, :, 0, 1], 1.0, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], g["noncausal_LSE"], atol=1e-12)
    O, L = ref(q, k, v, True, g["scale"])
    i = np.arange(S)
    np.testing.assert_allclose(O[0, :, 0, 0], i / 2.0, atol=1e-10)
    np.testing.assert_allclose(L[0, 0], np.log(i + 1.0), atol=1e-12)


def pin_identical_keys(ref):
    """All keys equal -> uniform softmax: O = mean of visible V,
    LSE_i = z_i0 + ln |N_i|."""
    B, S, H, D = 1, 37, 2, 5
    q = _rand((B, S, H, D), 1, 2.0)
    k = np.repeat(_rand((B, 1, H, D), 2, 3.0), S, axis=1)
    v = _rand((B, S, H, D), 3)
    scale = 0.3
    z0 = scale * np.einsum("bihd,bhd->bhi", q, k[:, 0])
    O, L = ref(q, k, v, False, scale)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=1, keepdims=True), O.shape),
                               atol=1e-12)
    np.testing.assert_allclose(L, z0 + math.log(S), atol=1e-12)
    O, L = ref(q, k, v, True, scale)
    prefix = np.cumsum(v, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    np.testing.assert_allclose(O, prefix, atol=1e-12)
    np.testing.assert_allclose(L, z0 + np.log(np.arange(1, S + 1))[None, None, :],
                               atol=1e-12)


def pin_causal_row0(ref):
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = z_00."""
    q, k, v = (_rand((2, 19, 3, 8), s) for s in (4, 5, 6))
    scale = 0.25
    O, L = ref(q, k, v, True, scale)
    np.testing.assert_allclose(O[:, 0], v[:, 0], atol=1e-13)
    np.testing.assert_allclose(L[:, :, 0], scale * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]),
                               atol=1e-13)


def pin_single_key(ref):
    """S = 1: O = V_0 and LSE = z_00 in both modes."""
    q, k, v = (_rand((3, 1, 2, 4), s) for s in (7, 8, 9))
    for causal in (False, True):
        O, L = ref(q, k, v, causal, 0.5)
        np.testing.assert_allclose(O, v, atol=1e-14)
        np.testing.assert_allclose(L[:, :, 0], 0.5 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]),
                                   atol=1e-14)


def pin_vanishing_scale(ref):
    """scale -> 0+: softmax -> uniform, O -> mean of visible V (error O(scale))."""
    q, k, v = (_rand((1, 23, 2, 6), s) for s in (10, 11, 12))
    O, L = ref(q, k, v, False, 1e-12)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(axis=1, keepdims=True), O.shape),
                               atol=1e-9)
    np.testing.assert_allclose(L, math.log(23), atol=1e-9)
    O, _ = ref(q, k, v, True, 1e-12)
    prefix = np.cumsum(v, axis=1) / np.arange(1, 24)[None, :, None, None]
    np.testing.assert_allclose(O, prefix, atol=1e-9)


def pin_dominant_key(ref):
    """One key's logit 40 above every other: O = V[j*] up to S*e^-40."""
    S, jstar = 29, 17
    q = np.ones((1, S, 1, 1))
    k = np.zeros((1, S, 1, 1))
    k[0, jstar, 0, 0] = 40.0 / 0.125
    v = _rand((1, S, 1, 3), 13)
    O, L = ref(q, k, v, False, 0.125)
    np.testing.assert_allclose(O[0, :, 0], np.broadcast_to(v[0, jstar, 0], (S, 3)),
                               atol=S * math.exp(-40) * 10)
    np.testing.assert_allclose(L[0, 0], 40.0 + math.log1p((S - 1) * math.exp(-40)),
                               atol=1e-12)


def pin_key_permutation(ref):
    """Non-causal attention is invariant under a joint permutation of K, V rows."""
    q, k, v = (_rand((1, 31, 2, 7), s) for s in (14, 15, 16))
    perm = np.random.default_rng(17).permutation(31)
    O1, L1 = ref(q, k, v, False, 0.4)
    O2, L2 = ref(q, k[:, perm], v[:, perm], False, 0.4)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def pin_lse_bounds(ref):
    """max_j z_ij <= LSE_i <= max_j z_ij + ln |N_i|."""
    q, k, v = (_rand((2, 40, 2, 8), s, 3.0) for s in (18, 19, 20))
    scale = 0.2
    for causal in (False, True):
        _, L = ref(q, k, v, causal, scale)
        z = scale * np.einsum("bihd,bjhd->bhij", q, k)
        n = np.arange(1, 41) if causal else np.full(40, 40)
        if causal:
            z = np.where(np.tril(np.ones((40, 40), bool)), z, -np.inf)
        zmax = z.max(axis=-1)
        assert np.all(L >= zmax - 1e-12)
        assert np.all(L <= zmax + np.log(n) + 1e-12)


def pin_torch_sdpa(ref):
    """Agreement with torch's own attention and logsumexp (fp64, CPU)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    q, k, v = (_rand((2, 45, 3, 16), s, 2.0) for s in (21, 22, 23))
    scale = 0.17
    for causal in (False, True):
        O, L = ref(q, k, v, causal, scale)
        tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            to = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
        np.testing.assert_allclose(O, to.permute(0, 2, 1, 3).numpy(), atol=1e-12)
        logits = scale * (tq @ tk.transpose(-1, -2))
        if causal:
            logits = logits.masked_fill(~torch.ones(45, 45, dtype=torch.bool).tril(), -math.inf)
        np.testing.assert_allclose(L, torch.logsumexp(logits, dim=-1).numpy(), atol=1e-12)


def pin_brute_force(ref):
    """Tiny inputs against a scalar loop with math.exp and exact summation."""
    for (S, D, causal, seed) in [(1, 1, False, 30), (2, 1, True, 31), (3, 2, False, 32),
                                 (4, 3, True, 33), (5, 2, True, 34), (5, 4, False, 35)]:
        q, k, v = (_rand((1, S, 2, D), seed + 100 * t) for t in range(3))
        scale = 0.6
        O, L = ref(q, k, v, causal, scale)
        for h in range(2):
            for i in range(S):
                keys = range(i + 1) if causal else range(S)
                z = [scale * math.fsum(q[0, i, h, d] * k[0, j, h, d] for d in range(D))
                     for j in keys]
                mz = max(z)
                w = [math.exp(x - mz) for x in z]
                tot = math.fsum(w)
                for d in range(D):
                    o = math.fsum(w[n] * v[0, j, h, d] for n, j in enumerate(keys)) / tot
                    assert abs(O[0, i, h, d] - o) < 1e-13
                assert abs(L[0, h, i] - (mz + math.log(tot))) < 1e-13


PINS = [pin_golden_worked_example, pin_uniform_scores, pin_identical_keys,
        pin_causal_row0, pin_single_key, pin_vanishing_scale, pin_dominant_key,
        pin_key_permutation, pin_lse_bounds, pin_torch_sdpa, pin_brute_force]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_reference_definition(pin):
    pin(attention_reference_f64)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("block,tau", [(1, 0.0), (3, 0.0), (3, 8 * math.log(2)),
                                       (16, 8 * math.log(2))])
def test_online_recurrence(pin, block, tau):
    """The pages' recurrence (with and without the lazy threshold) passes the
    same pins as the definition."""
    def ref(q, k, v, causal, scale):
        return online_softmax_attention(q, k, v, causal, scale, block, tau)
    pin(ref)


# ---------------------------------------------------------------------------
# further checks of individual pieces

def test_golden_online_trace():
    """The online state after each tile matches the hand-derived values."""
    g = _parse_golden("worked_example_two_tiles.txt")
    q = np.array(g["q"]).reshape(1, 4, 1, 1)
    k = np.array(g["k"]).reshape(1, 4, 1, 1)
    v = np.array(g["v"]).reshape(1, 4, 1, 1)
    trace = []
    online_softmax_attention(q, k, v, False, g["scale"], int(g["online_block"]), 0.0, trace)
    (t0, m0, l0, o0), (t1, m1, l1, o1) = trace
    assert abs(m0 - g["online_tile0_m"]) < 1e-14 and abs(l0 - g["online_tile0_l"]) < 1e-14
    assert abs(o0[0] - g["online_tile0_o"]) < 1e-13
    assert abs(m1 - g["online_tile1_m"]) < 1e-14 and abs(l1 - g["online_tile1_l"]) < 1e-14
    assert abs(o1[0] - g["online_tile1_o"]) < 1e-13


def test_rows_of_p_sum_to_one():
    for w in ("stress",):
        for causal in (False, True):
            q, k, _ = (_rand((1, 200, 2, 16), s, 4.0) for s in (40, 41, 42))
            for h in range(2):
                P = softmax_probabilities(q, k, causal, 0.125, 0, h)
                np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
                assert np.all(P >= 0)
                if causal:
                    assert np.all(np.triu(P, 1) == 0)


@pytest.mark.parametrize("block,tau,n_tiles", [(128, 8 * math.log(2), True),
                                               (64, 0.0, True), (128, 0.0, False)])
def test_online_matches_definition_on_workload_shapes(block, tau, n_tiles):
    """Tile size of the GPU kernel, a ragged length, masked tiles, peaky logits."""
    rng = np.random.default_rng(50)
    S, D = 300, 64
    q = rng.standard_normal((1, S, 1, D)) * 4
    k = rng.standard_normal((1, S, 1, D)) * 4
    v = rng.uniform(-1, 1, (1, S, 1, D))
    for causal in (False, True):
        O, L = attention_reference_f64(q, k, v, causal, 0.125)
        nt = (S + block - 1) // block if n_tiles else None
        O2, L2 = online_softmax_attention(q, k, v, causal, 0.125, block, tau, n_tiles=nt)
        np.testing.assert_allclose(O2, O, atol=1e-12)
        np.testing.assert_allclose(L2, L, rtol=1e-13, atol=1e-12)


def _half_by_formula(bits):
    s = -1.0 if bits >> 15 else 1.0
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    if e == 0:
        return s * math.ldexp(f, -24)
    if e == 31:
        return s * math.inf if f == 0 else math.nan
    return s * math.ldexp(1024 + f, e - 25)


def _bf16_by_formula(bits):
    s = -1.0 if bits >> 15 else 1.0
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0:
        return s * math.ldexp(f, -133)
    if e == 255:
        return s * math.inf if f == 0 else math.nan
    return s * math.ldexp(128 + f, e - 134)


def test_decoders_exact_on_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = decode_f16(bits)
    b = decode_bf16(bits)
    eh = np.array([_half_by_formula(int(x)) for x in range(65536)])
    eb = np.array([_bf16_by_formula(int(x)) for x in range(65536)])
    np.testing.assert_array_equal(np.isnan(h), np.isnan(eh))
    np.testing.assert_array_equal(h[~np.isnan(h)], eh[~np.isnan(eh)])
    np.testing.assert_array_equal(np.isnan(b), np.isnan(eb))
    np.testing.assert_array_equal(b[~np.isnan(b)], eb[~np.isnan(eb)])
    torch = pytest.importorskip("torch")
    tb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(tb), np.isnan(b))
    np.testing.assert_array_equal(tb[~np.isnan(tb)], b[~np.isnan(b)])


def test_bit_entry_points_match_float_path():
    """attention_reference / attention_rows decode the same values the float
    path sees, for both 16-bit types."""
    for dtype in ("f16", "bf16"):
        qb, kb, vb = fa_inputs.make_qkv(2, 3, 70, 16, dtype, "stress", 7,
                                        identical_key_head=(1, 2))
        dec = decode_f16 if dtype == "f16" else decode_bf16
        for causal in (False, True):
            O, L = attention_reference(qb, kb, vb, dtype, causal, 0.25)
            O2, L2 = attention_reference_f64(dec(qb), dec(kb), dec(vb), causal, 0.25)
            np.testing.assert_array_equal(O, O2)
            np.testing.assert_array_equal(L, L2)
            rows = [0, 5, 69]
            Or, Lr = attention_rows(qb, kb, vb, dtype, causal, 0.25, 1, 2, rows)
            np.testing.assert_allclose(Or, O[1, rows, 2, :], atol=1e-14)
            np.testing.assert_allclose(Lr, L[1, 2, rows], atol=1e-13)


def test_stress_identical_key_head_closed_form():
    """On the stress workload's identical-key head the oracle gives the mean /
    prefix mean of V (the closed form), at a reduced length."""
    qb, kb, vb = fa_inputs.make_qkv(3, 8, 150, 64, "f16", "stress", 1005,
                                    identical_key_head=(2, 7))
    v = decode_f16(vb)[2, :, 7, :]
    for causal in (False, True):
        O, _ = attention_reference(qb, kb, vb, "f16", causal, 0.125)
        if causal:
            want = np.cumsum(v, axis=0) / np.arange(1, 151)[:, None]
        else:
            want = np.broadcast_to(v.mean(axis=0), v.shape)
        np.testing.assert_allclose(O[2, :, 7, :], want, atol=1e-12)


# ---------------------------------------------------------------------------
# planted mistakes: every plausible slip in the oracle must fail some pin

def _mutant(kind):
    def ref(q, k, v, causal, scale):
        q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
        B, S, H, D = q.shape
        O = np.empty((B, S, H, v.shape[3])); L = np.empty((B, H, S))
        for b in range(B):
            for h in range(H):
                qh, kh, vh = q[b, :, h], k[b, :, h], v[b, :, h]
                sc = {"no_scale": 1.0, "scale_twice": scale * scale}.get(kind, scale)
                z = sc * (qh @ kh.T)
                if kind == "transposed":
                    z = sc * (kh @ qh.T)
                i = np.arange(S)[:, None]; j = np.arange(S)[None, :]
                vis = {"mask_flipped": j >= i, "mask_strict": j < i,
                       }.get(kind, j <= i) if causal else np.ones((S, S), bool)
                if kind == "mask_strict":
                    vis = vis | ((i == 0) & (j == 0))
                z = np.where(vis, z, -np.inf)
                m = z.max(axis=1)
                e = np.exp(z - m[:, None])
                l = e.sum(axis=1)
                p = e / l[:, None]
                if kind == "norm_wrong_axis":
                    p = e / np.maximum(e.sum(axis=0, keepdims=True), 1e-300)
                o = p @ vh
                if kind == "o_unnormalised":
                    o = e @ vh
                lse = m + np.log(l)
                if kind == "lse_no_max":
                    lse = np.log(l)
                if kind == "lse_log2":
                    lse = m + np.log2(l)
                O[b, :, h] = o; L[b, h] = lse
        return O, L
    return ref


def _online_mutant(kind):
    def ref(q, k, v, causal, scale):
        q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
        B, S, H, D = q.shape
        O = np.empty((B, S, H, v.shape[3])); L = np.empty((B, H, S))
        for b in range(B):
            for h in range(H):
                for i in range(S):
                    m, l, o = -math.inf, 0.0, np.zeros(v.shape[3])
                    last = i if causal else S - 1
                    for j0 in range(0, last + 1, 2):
                        j1 = min(last + 1, j0 + 2)
                        s = scale * (k[b, j0:j1, h] @ q[b, i, h])
                        m_new = max(m, s.max())
                        alpha = math.exp(m - m_new) if m > -math.inf else 0.0
                        p = np.exp(s - m_new)
                        l = (l if kind == "l_not_rescaled" else alpha * l) + p.sum()
                        o = (o if kind == "o_not_rescaled" else alpha * o) + p @ v[b, j0:j1, h]
                        m = m_new
                    O[b, i, h] = o / l
                    L[b, h, i] = m + math.log(l)
        return O, L
    return ref


MUTANTS = ["no_scale", "scale_twice", "transposed", "mask_flipped", "mask_strict",
           "norm_wrong_axis", "o_unnormalised", "lse_no_max", "lse_log2"]


def _fails_some_pin(ref):
    failed = []
    for pin in PINS:
        try:
            pin(ref)
        except AssertionError:
            failed.append(pin.__name__)
        except (ValueError, FloatingPointError, IndexError):
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes_every_pin():
    assert _fails_some_pin(_mutant("none")) == []
    assert _fails_some_pin(_online_mutant("none")) == []


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistakes(kind):
    assert _fails_some_pin(_mutant(kind)), f"no pin caught the planted mistake {kind}"


@pytest.mark.parametrize("kind", ["o_not_rescaled", "l_not_rescaled"])
def test_pins_catch_planted_recurrence_mistakes(kind):
    assert _fails_some_pin(_online_mutant(kind)), kind


# ------------------------------------------------------ grouped K/V heads
# Reading (not on the pages): with H_kv K/V heads, query head h uses K/V head
# h // (H / H_kv).  The pins below fix that grouping and reduce the grouped
# call to the single-head definition pinned above.

def test_grouped_heads_constant_values_pick_the_group():
    """V constant per K/V head (head j holds (j + 1) / 4 everywhere): every
    output of query head h equals the constant of its group's K/V head, which
    distinguishes h // group from any other assignment (h mod H_kv, ...)."""
    B, H, H_kv, S, D = 1, 6, 3, 37, 64
    rng = np.random.default_rng(21)
    q = rng.standard_normal((B, S, H, D))
    k = rng.standard_normal((B, S, H_kv, D))
    v = np.empty((B, S, H_kv, D))
    for j in range(H_kv):
        v[:, :, j, :] = (j + 1) / 4.0
    for causal in (False, True):
        O, _ = attention_reference_f64(q, k, v, causal, 0.125)
        for h in range(H):
            want = (h // (H // H_kv) + 1) / 4.0
            assert np.abs(O[:, :, h, :] - want).max() < 1e-12, (h, causal)


@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2), (6, 1), (8, 2)])
def test_grouped_heads_equal_single_head_calls(H, H_kv):
    """Each query head of a grouped call equals the single-head definition
    called on that head and its K/V head (MQA when H_kv = 1, MHA when equal)."""
    qb, kb, vb = fa_inputs.make_qkv(2, H, 45, 64, "f16", "normal", 22, h_kv=H_kv)
    for causal in (False, True):
        O, L = attention_reference(qb, kb, vb, "f16", causal, 0.125)
        for h in range(H):
            hk = h * H_kv // H
            o1, l1 = attention_reference(qb[:, :, h:h + 1], kb[:, :, hk:hk + 1], vb[:, :, hk:hk + 1],
                                         "f16", causal, 0.125)
            assert np.array_equal(O[:, :, h:h + 1], o1) and np.array_equal(L[:, h:h + 1], l1)


def test_grouped_heads_rows_match_full_reference():
    qb, kb, vb = fa_inputs.make_qkv(1, 8, 70, 64, "bf16", "stress", 23, h_kv=2)
    O, L = attention_reference(qb, kb, vb, "bf16", True, 0.125)
    rows = [0, 1, 33, 69]
    for h in (0, 3, 4, 7):
        o, l = attention_rows(qb, kb, vb, "bf16", True, 0.125, 0, h, rows)
        assert np.allclose(o, O[0, rows, h, :], rtol=0, atol=1e-13)
        assert np.allclose(l, L[0, h, rows], rtol=0, atol=1e-13)


def test_grouped_heads_must_divide():
    qb, kb, vb = fa_inputs.make_qkv(1, 4, 16, 64, "f16", "normal", 24, h_kv=3)
    with pytest.raises(ValueError):
        attention_reference(qb, kb, vb, "f16", False, 0.125)


# ------------------------------------------------------ variable length
# Reading (not on the pages): packed sequences, offsets cu, each sequence
# attends within itself; LSE is [H, total].

def test_varlen_equal_lengths_equal_the_batched_definition():
    """B sequences of one length packed back to back give the batched result
    (the [B, S, H, D] layout is the same memory with cu = 0, S, 2S, ...)."""
    B, S, H, D = 3, 70, 4, 64
    qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, "f16", "normal", 31, h_kv=2)
    cu = np.arange(B + 1, dtype=np.int32) * S
    for causal in (False, True):
        O, L = attention_reference(qb, kb, vb, "f16", causal, 0.125)
        Ov, Lv = attention_reference_varlen(qb.reshape(B * S, H, D), kb.reshape(B * S, 2, D),
                                            vb.reshape(B * S, 2, D), cu, "f16", causal, 0.125)
        assert np.array_equal(Ov, O.reshape(B * S, H, D))
        assert np.array_equal(Lv, L.transpose(1, 0, 2).reshape(H, B * S))


def test_varlen_sequences_do_not_see_each_other():
    """Changing every token of the other sequences leaves a sequence's output
    unchanged; the first row of a causal sequence equals its own V row 0."""
    lens = [5, 130, 1, 77]
    qb, kb, vb, cu = fa_inputs.make_varlen(lens, 2, 64, "bf16", "normal", 32)
    O, L = attention_reference_varlen(qb, kb, vb, cu, "bf16", True, 0.125)
    a, e = int(cu[1]), int(cu[2])
    q2, k2, v2, _ = fa_inputs.make_varlen(lens, 2, 64, "bf16", "normal", 33)
    for x, y in ((q2, qb), (k2, kb), (v2, vb)):
        x[a:e] = y[a:e]
    O2, L2 = attention_reference_varlen(q2, k2, v2, cu, "bf16", True, 0.125)
    assert np.array_equal(O2[a:e], O[a:e]) and np.array_equal(L2[:, a:e], L[:, a:e])
    assert not np.array_equal(O2[:a], O[:a])
    for b in range(len(lens)):
        r = int(cu[b])
        assert np.allclose(O[r], decode_bf16(vb[r]), rtol=0, atol=1e-12)   # causal row 0 = V[0]


def test_varlen_empty_sequences_and_bad_offsets():
    qb, kb, vb, cu = fa_inputs.make_varlen([0, 9, 0, 4], 1, 64, "f16", "normal", 34)
    O, L = attention_reference_varlen(qb, kb, vb, cu, "f16", False, 0.125)
    assert O.shape == (13, 1, 64) and np.all(np.isfinite(L))
    with pytest.raises(ValueError):
        attention_reference_varlen(qb, kb, vb, np.array([0, 9, 4, 13]), "f16", False, 0.125)


# ------------------------------------------------------ local (sliding window)
# Reading (not on the pages beyond "causal/local mask"): window (left, right)
# keeps key j for query i iff i - left <= j <= i + right (-1: no bound).

def _f64(bits, dtype="f16"):
    return decode_f16(bits) if dtype == "f16" else decode_bf16(bits)


def test_window_zero_width_returns_own_value():
    """(0, 0): every row sees only its own key, so O = V row by row and
    LSE = scale * q_i . k_i."""
    qb, kb, vb = fa_inputs.make_qkv(2, 3, 50, 64, "f16", "normal", 41)
    for causal in (False, True):
        O, L = attention_reference(qb, kb, vb, "f16", causal, 0.125, window=(0, 0))
        assert np.array_equal(O, _f64(vb))
        z = 0.125 * np.einsum("bshd,bshd->bhs", _f64(qb), _f64(kb))
        assert np.allclose(L, z, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", [(True, (1, -1)), (False, (1, 0)), (False, (1, 1))])
def test_window_of_two_or_three_keys_closed_form(causal, window):
    """Left bound 1 (causal, or right bound 0): keys {i-1, i}; window (1, 1):
    keys {i-1, i, i+1} -- a softmax over two or three logits written out."""
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 40, 64, "bf16", "stress", 42)
    q, k, v = _f64(qb, "bf16"), _f64(kb, "bf16"), _f64(vb, "bf16")
    O, L = attention_reference(qb, kb, vb, "bf16", causal, 0.125, window=window)
    S = 40
    right = 0 if (causal or window[1] == 0) else window[1]
    for h in range(2):
        for i in range(S):
            keys = [j for j in (i - 1, i, i + 1) if 0 <= j < S and i - 1 <= j <= i + right]
            z = np.array([0.125 * q[0, i, h] @ k[0, j, h] for j in keys])
            w = np.exp(z - z.max())
            o = sum(wj * v[0, j, h] for wj, j in zip(w, keys)) / w.sum()
            assert np.allclose(O[0, i, h], o, rtol=0, atol=1e-12)
            assert abs(L[0, h, i] - (z.max() + math.log(w.sum()))) < 1e-12


def test_unbounded_or_covering_window_is_the_plain_definition():
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 70, 64, "f16", "normal", 43)
    for causal in (False, True):
        O, L = attention_reference(qb, kb, vb, "f16", causal, 0.125)
        for window in ((-1, -1), (69, 69), (1000, -1), (-1, 1000)):
            Ow, Lw = attention_reference(qb, kb, vb, "f16", causal, 0.125, window=window)
            assert np.array_equal(Ow, O) and np.array_equal(Lw, L), (causal, window)


def test_window_rows_match_full_reference():
    qb, kb, vb = fa_inputs.make_qkv(1, 4, 300, 64, "f16", "normal", 44, h_kv=2)
    O, L = attention_reference(qb, kb, vb, "f16", True, 0.125, window=(37, -1))
    rows = [0, 5, 36, 37, 38, 299]
    o, l = attention_rows(qb, kb, vb, "f16", True, 0.125, 0, 3, rows, window=(37, -1))
    assert np.array_equal(o, O[0, rows, 3]) and np.array_equal(l, L[0, 3, rows])


# ------------------------------------------------------ dropout
from oracle import (attention_reference_dropout, dropout_keep, dropout_threshold,  # noqa: E402
                    philox4x32_10)


@pytest.mark.parametrize("ctr,key,want", [
    ((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff,) * 4, (0xffffffff,) * 2, (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
])
def test_philox_known_answer_vectors(ctr, key, want):
    """Philox4x32-10 against the known-answer vectors published with the
    generator (Random123 distribution)."""
    got = philox4x32_10(*[np.array([c]) for c in ctr], *key)
    assert tuple(int(w[0]) for w in got) == want


def test_dropout_mask_elements_one_by_one():
    """Element (b, h, i, j) of the mask, from one Philox call each: counter
    (j div 8, i, h, b), word (j mod 8) div 2, low half for even j; kept iff the
    half >= floor(p 2^16).  Catches a transposed or mis-strided layout."""
    B, H, S, p, seed = 2, 3, 77, 0.37, 0xFEDC_BA98_7654_3210
    keep = dropout_keep(B, H, S, p, seed)
    t = math.floor(p * 65536)
    rng = np.random.default_rng(3)
    for _ in range(300):
        b, h, i, j = (int(rng.integers(n)) for n in (B, H, S, S))
        words = philox4x32_10(np.array([j // 8]), np.array([i]), np.array([h]), np.array([b]),
                              seed % 2**32, seed // 2**32)
        w = int(words[(j % 8) // 2][0])
        half = (w >> 16) if j % 2 else (w & 0xFFFF)
        assert keep[b, h, i, j] == (half >= t), (b, h, i, j)


def test_dropout_threshold_quantisation():
    """p is taken to floor(p 2^16) / 2^16: p = 0.5 drops exactly the draws
    below 32768, and every p < 1 keeps the draw 65535."""
    assert dropout_threshold(0.0) == 0 and dropout_threshold(0.5) == 32768
    assert dropout_threshold(1.0 - 2.0 ** -20) == 65535
    assert dropout_threshold(0.1) == 6553


def test_dropout_zero_probability_is_the_plain_definition():
    qb, kb, vb = fa_inputs.make_qkv(1, 3, 90, 64, "f16", "normal", 51, h_kv=1)
    for causal in (False, True):
        O, L = attention_reference(qb, kb, vb, "f16", causal, 0.125)
        Od, Ld = attention_reference_dropout(qb, kb, vb, "f16", causal, 0.125, 0.0, 1234)
        assert np.allclose(Od, O, rtol=0, atol=1e-13) and np.array_equal(Ld, L)


def test_dropout_keeps_the_lse_and_the_expected_fraction():
    qb, kb, vb = fa_inputs.make_qkv(1, 2, 256, 64, "f16", "normal", 52)
    _, L = attention_reference(qb, kb, vb, "f16", True, 0.125)
    for p in (0.1, 0.5, 0.9):
        _, Ld = attention_reference_dropout(qb, kb, vb, "f16", True, 0.125, p, 99)
        assert np.array_equal(Ld, L)
        keep = dropout_keep(2, 3, 256, p, 7)
        n = keep.size
        assert abs(keep.mean() - (1 - p)) < 5 * math.sqrt(p * (1 - p) / n), p


def test_dropout_is_unbiased_over_seeds():
    """The mean of O over many seeds approaches the undropped O."""
    qb, kb, vb = fa_inputs.make_qkv(1, 1, 24, 64, "f16", "normal", 53)
    O, _ = attention_reference(qb, kb, vb, "f16", False, 0.125)
    acc = np.zeros_like(O)
    n = 400
    for s in range(n):
        acc += attention_reference_dropout(qb, kb, vb, "f16", False, 0.125, 0.3, 1000 + s)[0]
    assert np.abs(acc / n - O).max() < 0.06


def test_dropout_mask_read_back_through_one_hot_values():
    """V row j = e_j makes O[i, j] = P_ij keep_ij / (1 - p): the applied mask
    is exactly dropout_keep at (row i, key j) -- not its transpose."""
    S, D, p, seed = 48, 64, 0.4, 0x1234_5678_9ABC
    qb, kb, _ = fa_inputs.make_qkv(1, 2, S, D, "f16", "normal", 54)
    v = np.zeros((1, S, 2, D), dtype=np.float32)
    for j in range(S):
        v[0, j, :, j] = 1.0
    vb = fa_inputs.f32_to_bits(v, "f16")
    for causal in (False, True):
        O, _ = attention_reference_dropout(qb, kb, vb, "f16", causal, 0.125, p, seed)
        keep = dropout_keep(1, 2, S, p, seed)
        vis = np.tril(np.ones((S, S), dtype=bool)) if causal else np.ones((S, S), dtype=bool)
        for h in range(2):
            got = O[0, :, h, :S] != 0
            assert np.array_equal(got, keep[0, h] & vis), (causal, h)


# ------------------------------------------------------ other head dimensions
@pytest.mark.parametrize("D", [8, 40, 136, 256])
def test_head_dims_closed_forms_and_torch(D):
    """The definition at head dimensions the kernels take besides 64 / 128:
    identical keys give the (prefix) mean of V, causal row 0 gives V row 0
    with LSE = its own logit, and torch's math attention agrees in fp64."""
    torch = pytest.importorskip("torch")
    S, H = 37, 2
    qb, kb, vb = fa_inputs.make_qkv(1, H, S, D, "bf16", "normal", 500 + D)
    kb = kb.copy()
    kb[0, :, 1, :] = kb[0, 0, 1, :]                    # head 1: every key equals key 0
    q, k, v = (decode_bf16(x) for x in (qb, kb, vb))
    scale = D ** -0.5
    for causal in (False, True):
        O, L = attention_reference(qb, kb, vb, "bf16", causal, scale)
        v1 = v[0, :, 1, :]
        want = (np.cumsum(v1, axis=0) / np.arange(1, S + 1)[:, None]) if causal else \
            np.broadcast_to(v1.mean(axis=0), v1.shape)
        np.testing.assert_allclose(O[0, :, 1, :], want, atol=1e-12)
        if causal:
            np.testing.assert_allclose(O[0, 0, :, :], v[0, 0, :, :], atol=1e-12)
            z00 = scale * np.einsum("hd,hd->h", q[0, 0], k[0, 0])
            np.testing.assert_allclose(L[0, :, 0], z00, atol=1e-12)
        tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))) for x in (q, k, v))
        mask = torch.ones(S, S, dtype=torch.bool).tril() if causal else None
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(O, ref.numpy().transpose(0, 2, 1, 3), atol=1e-12)
