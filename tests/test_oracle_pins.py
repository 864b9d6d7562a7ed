"""Pins for the fp64 oracle, each against something other than the oracle itself.

Sources are the pages' definitions ("Attention Kernel 계보": p.2 §1 attention,
p.3 §2-§9 softmax passes and LSE, p.4 merge, p.13 causal mask, p.15 GQA head
map), closed forms derived by hand (``tests/golden/closed_form.json``),
invariants of softmax, and an independent brute force in decimal arithmetic.
Each pin is chosen so that a plausible slip in the oracle (dropped m in LSE,
wrong head map, off-by-one causal bound, missing scale, transposed operand,
lost merge factor) fails at least one of them.
"""
import decimal
import json
import math
import os

import numpy as np
import pytest
import torch

from gqa_attention_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")
TOL = 1e-12


def _ev(expr):
    return float(eval(str(expr), {"__builtins__": {}}, {"ln": math.log, "nan": math.nan,
                                                          "inf": math.inf}))


def _arr(nested):
    if isinstance(nested, list):
        return np.array([_arr(x) for x in nested], dtype=np.float64)
    return _ev(nested)


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


# ---------------------------------------------------------------- golden ---
def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_closed_forms(oracle_mod, case):
    if case["kind"] == "merge":
        out, lse = oracle_mod.merge_partials(_arr(case["m"]), _arr(case["l"]), _arr(case["O"]))
    elif case["kind"] == "chunk":
        out, lse = oracle_mod.prefill_chunk_rows(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]),
                                                 _ev(case["scale"]), seq_lens=case["seq_lens"],
                                                 window=case["window"])
    elif case["kind"] == "decode":
        out, lse = oracle_mod.decode(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]),
                                     case["seq_lens"], _ev(case["scale"]))
    else:
        out, lse = oracle_mod.prefill_causal_rows(_arr(case["q"]), _arr(case["k"]),
                                                  _arr(case["v"]), _ev(case["scale"]))
    np.testing.assert_allclose(out, _arr(case["out"]), rtol=TOL, atol=TOL)
    np.testing.assert_allclose(lse, _arr(case["lse"]), rtol=TOL, atol=TOL)


# ----------------------------------------------------------- closed forms ---
def test_single_key_returns_that_value(oracle_mod):
    rng = np.random.default_rng(1)
    B, H_q, H_kv, d, S = 2, 6, 3, 16, 5
    q, k, v = _rand((B, H_q, d), rng), _rand((B, S, H_kv, d), rng), _rand((B, S, H_kv, d), rng)
    tau = 0.3
    out, lse = oracle_mod.decode(q, k, v, [1, 1], tau)
    G = H_q // H_kv
    for b in range(B):
        for h in range(H_q):
            np.testing.assert_allclose(out[b, h], v[b, 0, h // G], rtol=0, atol=1e-13)
            assert lse[b, h] == pytest.approx(tau * q[b, h] @ k[b, 0, h // G], abs=1e-13)


def test_identical_keys_give_mean_of_values(oracle_mod):
    rng = np.random.default_rng(2)
    B, H_q, H_kv, d, S = 1, 4, 2, 8, 37
    q = _rand((B, H_q, d), rng)
    k = np.broadcast_to(_rand((B, 1, H_kv, d), rng), (B, S, H_kv, d)).copy()
    v = _rand((B, S, H_kv, d), rng)
    tau = 1 / math.sqrt(d)
    out, lse = oracle_mod.decode(q, k, v, [S], tau)
    for h in range(H_q):
        kv = h // 2
        np.testing.assert_allclose(out[0, h], v[0, :, kv].mean(axis=0), atol=1e-13)
        assert lse[0, h] == pytest.approx(tau * q[0, h] @ k[0, 0, kv] + math.log(S), abs=1e-12)


def test_zero_query_is_uniform_over_visible_keys(oracle_mod):
    rng = np.random.default_rng(3)
    B, S, H_q, H_kv, d = 2, 23, 4, 1, 8
    q = np.zeros((B, S, H_q, d))
    k, v = _rand((B, S, H_kv, d), rng), _rand((B, S, H_kv, d), rng)
    out, lse = oracle_mod.prefill_causal_rows(q, k, v, 0.7)
    for i in range(S):
        np.testing.assert_allclose(out[:, i, :, :], np.broadcast_to(
            v[:, : i + 1, 0, :].mean(axis=1)[:, None, :], (B, H_q, d)), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(i + 1), atol=1e-13)
    # decode: LSE = ln L_b and O = mean of the first L_b values
    qd = np.zeros((B, H_q, d))
    out, lse = oracle_mod.decode(qd, k, v, [5, 23], 0.7)
    np.testing.assert_allclose(lse[0], math.log(5), atol=1e-13)
    np.testing.assert_allclose(lse[1], math.log(23), atol=1e-13)
    np.testing.assert_allclose(out[1, 2], v[1, :, 0].mean(axis=0), atol=1e-13)


def test_causal_row_zero_is_first_value(oracle_mod):
    rng = np.random.default_rng(4)
    B, S, H_q, H_kv, d = 1, 9, 8, 2, 16
    q, k, v = (_rand((B, S, H_q, d), rng), _rand((B, S, H_kv, d), rng),
               _rand((B, S, H_kv, d), rng))
    out, lse = oracle_mod.prefill_causal_rows(q, k, v, 0.25, rows=[0])
    for h in range(H_q):
        np.testing.assert_allclose(out[0, 0, h], v[0, 0, h // 4], atol=1e-14)
        assert lse[0, h, 0] == pytest.approx(0.25 * q[0, 0, h] @ k[0, 0, h // 4], abs=1e-13)


# ------------------------------------------------------------- invariants ---
def test_gqa_equals_mha_with_repeated_kv_heads(oracle_mod):
    rng = np.random.default_rng(5)
    B, S, H_q, H_kv, d = 2, 19, 12, 3, 8
    G = H_q // H_kv
    q, k, v = (_rand((B, S, H_q, d), rng), _rand((B, S, H_kv, d), rng),
               _rand((B, S, H_kv, d), rng))
    out_g, lse_g = oracle_mod.prefill_causal_rows(q, k, v, 0.4)
    out_m, lse_m = oracle_mod.prefill_causal_rows(q, np.repeat(k, G, axis=2),
                                                  np.repeat(v, G, axis=2), 0.4)
    np.testing.assert_allclose(out_g, out_m, atol=1e-14)
    np.testing.assert_allclose(lse_g, lse_m, atol=1e-14)
    qd = q[:, 0]
    out_g, lse_g = oracle_mod.decode(qd, k, v, [7, 19], 0.4)
    out_m, lse_m = oracle_mod.decode(qd, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2),
                                     [7, 19], 0.4)
    np.testing.assert_allclose(out_g, out_m, atol=1e-14)
    np.testing.assert_allclose(lse_g, lse_m, atol=1e-14)


@pytest.mark.parametrize("chunk", [1, 3, 8, 64, 1000])
def test_split_then_merge_equals_unsplit(oracle_mod, chunk):
    rng = np.random.default_rng(6)
    B, S, H_q, H_kv, d = 3, 50, 4, 2, 8
    q, k, v = _rand((B, H_q, d), rng), _rand((B, S, H_kv, d), rng, 2.0), _rand((B, S, H_kv, d), rng)
    lens = [50, 1, 33]
    n_split = -(-S // chunk)
    m, l, O = oracle_mod.decode_partials(q, k, v, lens, 0.35, n_split, chunk)
    out_s, lse_s = oracle_mod.merge_partials(m, l, O)
    out, lse = oracle_mod.decode(q, k, v, lens, 0.35)
    np.testing.assert_allclose(out_s, out, atol=1e-12)
    np.testing.assert_allclose(lse_s, lse, atol=1e-12)
    # empty splits are the identity (-inf, 0)
    for b, L in enumerate(lens):
        for s_ in range(n_split):
            if s_ * chunk >= L:
                assert m[b, :, s_].tolist() == [-math.inf] * H_q
                assert (l[b, :, s_] == 0).all()


def test_merge_is_commutative_and_has_identity(oracle_mod):
    rng = np.random.default_rng(7)
    R, n, d = 5, 6, 4
    m = rng.standard_normal((R, n)) * 3
    l = rng.uniform(0.5, 4.0, (R, n))
    O = rng.standard_normal((R, n, d))
    out, lse = oracle_mod.merge_partials(m, l, O)
    perm = rng.permutation(n)
    out_p, lse_p = oracle_mod.merge_partials(m[:, perm], l[:, perm], O[:, perm])
    np.testing.assert_allclose(out_p, out, atol=1e-13)
    np.testing.assert_allclose(lse_p, lse, atol=1e-13)
    m_id = np.concatenate([m, np.full((R, 2), -np.inf)], axis=1)
    l_id = np.concatenate([l, np.zeros((R, 2))], axis=1)
    O_id = np.concatenate([O, np.zeros((R, 2, d))], axis=1)
    out_i, lse_i = oracle_mod.merge_partials(m_id, l_id, O_id)
    np.testing.assert_allclose(out_i, out, atol=1e-13)
    np.testing.assert_allclose(lse_i, lse, atol=1e-13)
    # closed form of the merge: LSE = ln sum_s l_s e^{m_s}; O = sum_s e^{m_s} O_s / sum_s l_s e^{m_s}
    w = np.exp(m)
    np.testing.assert_allclose(lse, np.log((l * w).sum(axis=1)), atol=1e-12)
    np.testing.assert_allclose(out, (w[:, :, None] * O).sum(1) / (l * w).sum(1)[:, None],
                               atol=1e-12)


def test_shift_of_keys_along_query_shifts_lse_only(oracle_mod):
    rng = np.random.default_rng(8)
    B, S, H_q, d = 1, 30, 1, 8
    q, k, v = _rand((B, 1, d), rng), _rand((B, S, 1, d), rng), _rand((B, S, 1, d), rng)
    lam, tau = 2.5, 0.3
    out0, lse0 = oracle_mod.decode(q, k, v, [S], tau)
    k2 = k + lam * q[:, None, :, :]
    out1, lse1 = oracle_mod.decode(q, k2, v, [S], tau)
    np.testing.assert_allclose(out1, out0, atol=1e-12)
    assert lse1[0, 0] - lse0[0, 0] == pytest.approx(tau * lam * float(q[0, 0] @ q[0, 0]),
                                                    abs=1e-11)


def test_decode_ignores_key_order(oracle_mod):
    rng = np.random.default_rng(9)
    S, d = 40, 16
    q, k, v = _rand((1, 2, d), rng), _rand((1, S, 1, d), rng), _rand((1, S, 1, d), rng)
    perm = rng.permutation(S)
    out0, lse0 = oracle_mod.decode(q, k, v, [S], 0.25)
    out1, lse1 = oracle_mod.decode(q, k[:, perm], v[:, perm], [S], 0.25)
    np.testing.assert_allclose(out1, out0, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0, atol=1e-13)


def test_prefill_row_equals_decode_on_its_prefix(oracle_mod):
    rng = np.random.default_rng(10)
    B, S, H_q, H_kv, d = 2, 21, 4, 2, 8
    q, k, v = (_rand((B, S, H_q, d), rng), _rand((B, S, H_kv, d), rng),
               _rand((B, S, H_kv, d), rng))
    rows = [0, 1, 7, 20]
    out, lse = oracle_mod.prefill_causal_rows(q, k, v, 0.5, rows=rows)
    for r, i in enumerate(rows):
        o_d, l_d = oracle_mod.decode(q[:, i], k, v, [i + 1] * B, 0.5)
        np.testing.assert_allclose(out[:, r], o_d, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, r], l_d, atol=1e-13)


def test_bf16_inputs_are_widened_exactly(oracle_mod):
    q, k, v, lens = inputs.decode_inputs(2, 4, 2, 16, 33, seed=3, seq_lens=[33, 10])
    out_b, lse_b = oracle_mod.decode(q, k, v, lens, 0.25)
    out_f, lse_f = oracle_mod.decode(q.double(), k.double(), v.double(), lens, 0.25)
    assert np.array_equal(out_b, out_f) and np.array_equal(lse_b, lse_f)
    assert np.isfinite(out_b).all()  # NaN padding past seq_lens is never read


# ------------------------------------------- independent re-derivations ---
def _brute_decimal(qrow, keys, vals, tau, prec=50):
    """Naive softmax attention of one row in decimal arithmetic (p.2 §1, p.3 §1).

    Inputs are converted to Decimal exactly; no max subtraction is needed since
    decimal exponents do not overflow at these magnitudes.
    """
    D = decimal.Decimal
    with decimal.localcontext() as ctx:
        ctx.prec = prec
        s = [D(float(tau)) * sum((D(float(a)) * D(float(b)) for a, b in zip(qrow, kj)), D(0))
             for kj in keys]
        e = [x.exp() for x in s]
        tot = sum(e, D(0))
        out = [float(sum((ei * D(float(vj[t])) for ei, vj in zip(e, vals)), D(0)) / tot)
               for t in range(len(vals[0]))]
        return out, float(tot.ln())


def test_brute_force_decimal_tiny_shapes(oracle_mod):
    rng = np.random.default_rng(11)
    B, S, H_q, H_kv, d = 2, 6, 4, 2, 3
    G = H_q // H_kv
    q, k, v = (_rand((B, S, H_q, d), rng), _rand((B, S, H_kv, d), rng, 1.5),
               _rand((B, S, H_kv, d), rng))
    tau = 0.6
    out, lse = oracle_mod.prefill_causal_rows(q, k, v, tau)
    for b in range(B):
        for i in range(S):
            for h in range(H_q):
                ref_o, ref_l = _brute_decimal(q[b, i, h], k[b, : i + 1, h // G],
                                              v[b, : i + 1, h // G], tau)
                np.testing.assert_allclose(out[b, i, h], ref_o, rtol=1e-13, atol=1e-14)
                assert lse[b, h, i] == pytest.approx(ref_l, rel=1e-13, abs=1e-14)
    lens = [6, 4]
    out, lse = oracle_mod.decode(q[:, 2], k, v, lens, tau)
    for b in range(B):
        for h in range(H_q):
            ref_o, ref_l = _brute_decimal(q[b, 2, h], k[b, : lens[b], h // G],
                                          v[b, : lens[b], h // G], tau)
            np.testing.assert_allclose(out[b, h], ref_o, rtol=1e-13, atol=1e-14)
            assert lse[b, h] == pytest.approx(ref_l, rel=1e-13, abs=1e-14)


def _online_two_pass(s, vals):
    """p.3 §4: streaming (m, l) in one pass, then the outputs in a second."""
    m, l = -math.inf, 0.0
    for x in s:
        m_new = max(m, x)
        l = l * math.exp(m - m_new) + math.exp(x - m_new)
        m = m_new
    o = sum(math.exp(x - m) / l * vj for x, vj in zip(s, vals))
    return o, m + math.log(l)


def _online_fused(s, vals):
    """p.3 §5: (m, l, O) streamed together, O rescaled whenever m grows, divided once."""
    m, l, o = -math.inf, 0.0, np.zeros_like(vals[0])
    for x, vj in zip(s, vals):
        m_new = max(m, x)
        corr = math.exp(m - m_new)
        l = l * corr + math.exp(x - m_new)
        o = o * corr + math.exp(x - m_new) * vj
        m = m_new
    return o / l, m + math.log(l)


def test_three_pass_matches_online_forms(oracle_mod):
    rng = np.random.default_rng(12)
    S, d, tau = 60, 8, 0.5
    q, k, v = _rand((1, 1, d), rng), _rand((1, S, 1, d), rng, 3.0), _rand((1, S, 1, d), rng)
    out, lse = oracle_mod.decode(q, k, v, [S], tau)
    s = [tau * float(q[0, 0] @ k[0, j, 0]) for j in range(S)]
    vals = [v[0, j, 0] for j in range(S)]
    for fn in (_online_two_pass, _online_fused):
        o, l_ = fn(s, vals)
        np.testing.assert_allclose(out[0, 0], o, atol=1e-12)
        assert lse[0, 0] == pytest.approx(l_, abs=1e-12)


# -------------------------------------------------------- argument checks ---
def test_invalid_arguments_raise(oracle_mod):
    q = np.zeros((1, 3, 4))
    k = np.zeros((1, 5, 2, 4))
    with pytest.raises(ValueError):
        oracle_mod.decode(q, k, k, [5], 1.0)  # H_q not a multiple of H_kv
    q = np.zeros((1, 4, 4))
    with pytest.raises(ValueError):
        oracle_mod.decode(q, k, k, [0], 1.0)  # empty sequence
    with pytest.raises(ValueError):
        oracle_mod.decode(q, k, k, [6], 1.0)  # longer than the cache
    with pytest.raises(ValueError):
        oracle_mod.prefill_causal_rows(np.zeros((1, 5, 4, 4)), k, k, 1.0, rows=[5])


# --------------------------------------------------------- input recipes ---
def test_input_generators_are_seeded_and_padded():
    a = inputs.decode_inputs(3, 8, 2, 32, 100, seed=5, ragged=(10, 100))
    b = inputs.decode_inputs(3, 8, 2, 32, 100, seed=5, ragged=(10, 100))
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
    q, k, v, lens = a
    assert q.dtype == torch.bfloat16 and lens.dtype == torch.int32
    for bb in range(3):
        L = int(lens[bb])
        assert 10 <= L <= 100
        assert torch.isfinite(k[bb, :L].float()).all() and torch.isnan(k[bb, L:].float()).all()
    rows = inputs.sample_rows(1000, 16, seed=0)
    assert rows[0] == 0 and rows[-1] == 999 and len(rows) == 16
    assert torch.equal(rows, inputs.sample_rows(1000, 16, seed=0))


# ------------------------------------------- chunked prefill, sliding window ---
def test_chunk_equal_to_full_prefill_when_it_is_the_whole_sequence(oracle_mod):
    rng = np.random.default_rng(20)
    B, S, H_q, H_kv, d = 2, 33, 4, 2, 8
    q, k, v = (_rand((B, S, H_q, d), rng), _rand((B, S, H_kv, d), rng),
               _rand((B, S, H_kv, d), rng))
    a_o, a_l = oracle_mod.prefill_causal_rows(q, k, v, 0.3)
    b_o, b_l = oracle_mod.prefill_chunk_rows(q, k, v, 0.3)
    np.testing.assert_allclose(b_o, a_o, atol=1e-14)
    np.testing.assert_allclose(b_l, a_l, atol=1e-14)


def test_chunk_rows_are_the_tail_rows_of_the_full_prefill(oracle_mod):
    rng = np.random.default_rng(21)
    B, S_max, T_q, H_q, H_kv, d = 2, 40, 7, 6, 3, 8
    lens = [40, 23]
    k, v = _rand((B, S_max, H_kv, d), rng), _rand((B, S_max, H_kv, d), rng)
    qc = _rand((B, T_q, H_q, d), rng)
    out, lse = oracle_mod.prefill_chunk_rows(qc, k, v, 0.4, seq_lens=lens)
    for b, L in enumerate(lens):
        qf = _rand((1, L, H_q, d), rng)
        qf[0, L - T_q:] = qc[b]
        f_o, f_l = oracle_mod.prefill_causal_rows(qf, k[b:b + 1, :L], v[b:b + 1, :L], 0.4,
                                                  rows=np.arange(L - T_q, L))
        np.testing.assert_allclose(out[b], f_o[0], atol=1e-13)
        np.testing.assert_allclose(lse[b], f_l[0], atol=1e-13)


def test_single_query_chunk_is_decode(oracle_mod):
    rng = np.random.default_rng(22)
    B, S_max, H_q, H_kv, d = 3, 50, 4, 1, 16
    k, v, q = _rand((B, S_max, H_kv, d), rng), _rand((B, S_max, H_kv, d), rng), _rand((B, H_q, d), rng)
    lens = [50, 1, 17]
    c_o, c_l = oracle_mod.prefill_chunk_rows(q[:, None], k, v, 0.25, seq_lens=lens)
    d_o, d_l = oracle_mod.decode(q, k, v, lens, 0.25)
    np.testing.assert_allclose(c_o[:, 0], d_o, atol=1e-14)
    np.testing.assert_allclose(c_l[:, :, 0], d_l, atol=1e-14)


def test_window_limits_and_closed_forms(oracle_mod):
    rng = np.random.default_rng(23)
    B, S, H_q, H_kv, d = 1, 30, 2, 1, 8
    q, k, v = (_rand((B, S, H_q, d), rng), _rand((B, S, H_kv, d), rng),
               _rand((B, S, H_kv, d), rng))
    full_o, full_l = oracle_mod.prefill_chunk_rows(q, k, v, 0.5)
    wide_o, wide_l = oracle_mod.prefill_chunk_rows(q, k, v, 0.5, window=S)
    np.testing.assert_allclose(wide_o, full_o, atol=1e-14)
    np.testing.assert_allclose(wide_l, full_l, atol=1e-14)
    # window 0: only the diagonal key
    o0, l0 = oracle_mod.prefill_chunk_rows(q, k, v, 0.5, window=0)
    for i in range(S):
        np.testing.assert_allclose(o0[0, i, 0], v[0, i, 0], atol=1e-14)
        assert l0[0, 0, i] == pytest.approx(0.5 * q[0, i, 0] @ k[0, i, 0], abs=1e-13)
    # zero queries: uniform over the window
    W = 5
    oz, lz = oracle_mod.prefill_chunk_rows(np.zeros_like(q), k, v, 0.5, window=W)
    for i in range(S):
        lo = max(0, i - W)
        np.testing.assert_allclose(oz[0, i, 1], v[0, lo:i + 1, 0].mean(axis=0), atol=1e-13)
        assert lz[0, 1, i] == pytest.approx(math.log(i + 1 - lo), abs=1e-13)


def test_window_brute_force_decimal(oracle_mod):
    rng = np.random.default_rng(24)
    B, S_max, T_q, H_q, H_kv, d, W = 1, 9, 4, 2, 1, 3, 2
    k, v = _rand((B, S_max, H_kv, d), rng), _rand((B, S_max, H_kv, d), rng)
    q = _rand((B, T_q, H_q, d), rng)
    out, lse = oracle_mod.prefill_chunk_rows(q, k, v, 0.7, seq_lens=[8], window=W)
    for i in range(T_q):
        a = 8 - T_q + i
        lo = max(0, a - W)
        for h in range(H_q):
            ref_o, ref_l = _brute_decimal(q[0, i, h], k[0, lo:a + 1, 0], v[0, lo:a + 1, 0], 0.7)
            np.testing.assert_allclose(out[0, i, h], ref_o, rtol=1e-13, atol=1e-14)
            assert lse[0, h, i] == pytest.approx(ref_l, rel=1e-13, abs=1e-14)


# ------------------------------------------------------------ paged decode ---
def _to_pages(k, B_p, rng, extra=3):
    """Scatter a contiguous cache [B, S, H, d] into a shuffled pool; returns (pool, table)."""
    B, S, H, d = k.shape
    nb = S // B_p
    perm = rng.permutation(B * nb + extra)  # physical page of each logical block
    pool = rng.standard_normal((B * nb + extra, B_p, H, d)) * 100  # unused pages: junk
    table = np.zeros((B, nb), dtype=np.int32)
    for b in range(B):
        for j in range(nb):
            p = perm[b * nb + j]
            pool[p] = k[b, j * B_p:(j + 1) * B_p]
            table[b, j] = p
    return pool, table


@pytest.mark.parametrize("B_p", [1, 4, 16])
def test_paged_decode_equals_contiguous_decode(oracle_mod, B_p):
    rng = np.random.default_rng(30 + B_p)
    B, S, H_q, H_kv, d = 3, 48, 8, 2, 8
    q, k, v = _rand((B, H_q, d), rng), _rand((B, S, H_kv, d), rng), _rand((B, S, H_kv, d), rng)
    lens = [48, 1, 29]
    kp, table = _to_pages(k, B_p, np.random.default_rng(5))
    vp, table_v = _to_pages(v, B_p, np.random.default_rng(5))
    assert np.array_equal(table, table_v)
    p_o, p_l = oracle_mod.decode_paged(q, kp, vp, table, lens, 0.3)
    c_o, c_l = oracle_mod.decode(q, k, v, lens, 0.3)
    np.testing.assert_allclose(p_o, c_o, atol=1e-14)
    np.testing.assert_allclose(p_l, c_l, atol=1e-14)


def test_paged_decode_shared_prefix_pages(oracle_mod):
    # two requests share their first two pages (copy-on-write prefix, p.17 §7)
    rng = np.random.default_rng(40)
    B_p, H_q, H_kv, d = 4, 4, 1, 8
    kp, vp = _rand((6, B_p, H_kv, d), rng), _rand((6, B_p, H_kv, d), rng)
    table = np.array([[3, 1, 5], [3, 1, 0]], dtype=np.int32)
    q = _rand((2, H_q, d), rng)
    q[1] = q[0]
    o, l_ = oracle_mod.decode_paged(q, kp, vp, table, [8, 8], 0.5)  # only the shared pages
    np.testing.assert_allclose(o[0], o[1], atol=0)
    np.testing.assert_allclose(l_[0], l_[1], atol=0)
    o2, _ = oracle_mod.decode_paged(q, kp, vp, table, [12, 12], 0.5)  # diverging third page
    assert not np.allclose(o2[0], o2[1])


def test_paged_decode_rejects_bad_pages(oracle_mod):
    kp = np.zeros((2, 4, 1, 8))
    with pytest.raises(ValueError):
        oracle_mod.decode_paged(np.zeros((1, 1, 8)), kp, kp, [[0, 2]], [8], 1.0)


# ------------------------------------------------------------- FP8 cache ---
def test_e4m3_decoding_matches_torch_for_every_code(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle_mod.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all() and nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(mine[~nan], ref[~nan])
    assert oracle_mod.e4m3_to_double(0x7E) == 448.0 and oracle_mod.e4m3_to_double(1) == 2.0 ** -9


def test_fp8_decode_equals_decode_of_the_dequantised_cache(oracle_mod):
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(2, 8, 2, 32, 40, seed=3, seq_lens=[40, 9])
    out8, lse8 = oracle_mod.decode_fp8(q, k8, v8, ks, vs, lens, 0.2)
    kd = k8.view(torch.float8_e4m3fn).double() * ks.double()[:, :, None, None]
    vd = v8.view(torch.float8_e4m3fn).double() * vs.double()[:, :, None, None]
    out, lse = oracle_mod.decode(q.double(), kd, vd, lens, 0.2)
    np.testing.assert_allclose(out8, out, atol=1e-14)
    np.testing.assert_allclose(lse8, lse, atol=1e-14)
    assert np.isfinite(out8).all()  # NaN codes and scales past seq_lens are never read
