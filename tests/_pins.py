"""Checks that pin the fp64 oracle to facts outside itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a value the pages print, a hand expansion, a closed
form, a special case that reduces to a library routine, or the invariant the
pages state (the parallel, recurrent and chunkwise forms give the same
output).  test_oracle.py runs them on the real oracle; test_oracle_mutants.py
runs them on copies with planted mistakes and expects at least one to fail.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(x) for x in rest])
    return vals


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _all_forms(o, q, k, v, g, chunks=()):
    """Outputs and final states of every form; chunkwise for each chunk size."""
    res = {"parallel": (o.parallel(q, k, v, g), None)}
    res["recurrent"] = o.recurrent(q, k, v, g)
    for C in chunks:
        res[f"chunk{C}"] = o.chunkwise(q, k, v, g, C)
    return res


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    scale = max(np.max(np.abs(b)), 1e-300) if b.size else 1.0
    err = np.max(np.abs(a - b)) / scale if a.size else 0.0
    assert err <= tol, f"{what}: normalised error {err:.3e} > {tol:.1e}"


# --- values the pages print ------------------------------------------------

def check_gamma_printed(o):
    """gamma_h = 1 - 2^(-5-h) (0-based h); the printed 0.996094 / ~177 tokens."""
    gold = _read_golden("decay_half_life.txt")
    assert o.gamma(0) == 0.96875 and o.gamma(1) == 0.984375
    g3 = o.gamma(3)
    assert g3 == 1.0 - 2.0 ** -8
    assert round(g3, 6) == gold["gamma_printed"][0]
    half_life = math.log(2.0) / -math.log(g3)
    assert round(half_life) == gold["half_life_tokens_printed"][0]
    hs = np.arange(16)
    assert np.array_equal(o.gamma(hs), 1.0 - 2.0 ** (-5.0 - hs))


# --- hand expansions ---------------------------------------------------------

def check_hand_expanded_scalar(o):
    gold = _read_golden("hand_expanded_n3.txt")
    q = gold["q"].reshape(1, 1, 3, 1)
    k = gold["k"].reshape(1, 1, 3, 1)
    v = gold["v"].reshape(1, 1, 3, 1)
    g = gold["gamma"]
    want_o = gold["out"].reshape(1, 1, 3, 1)
    want_s = gold["state"].reshape(1, 1, 1, 1)
    res = _all_forms(o, q, k, v, g, chunks=(1, 2, 3, 4))
    for name, (out, S) in res.items():
        assert np.array_equal(out, want_o), (name, out.ravel(), want_o.ravel())
        if S is not None:
            assert np.array_equal(S, want_s), (name, S.ravel())


def check_hand_expanded_vector(o):
    gold = _read_golden("hand_expanded_vec.txt")
    q = gold["q"].reshape(1, 1, 2, 2)
    k = gold["k"].reshape(1, 1, 2, 2)
    v = gold["v"].reshape(1, 1, 2, 2)
    g = gold["gamma"]
    want_o = gold["out_times_sqrt2"].reshape(1, 1, 2, 2) / math.sqrt(2.0)
    want_s = gold["state"].reshape(1, 1, 2, 2)
    res = _all_forms(o, q, k, v, g, chunks=(1, 2))
    for name, (out, S) in res.items():
        _close(out, want_o, 1e-15, name)
        if S is not None:
            assert np.array_equal(S, want_s), (name, S.ravel())


def check_one_step_from_state(o):
    """One recurrent step from a given state: S' = g S + k v, o = q S' (d = 1)."""
    q = np.array([4.0]).reshape(1, 1, 1, 1)
    k = np.array([3.0]).reshape(1, 1, 1, 1)
    v = np.array([-1.0]).reshape(1, 1, 1, 1)
    S0 = np.array([2.0]).reshape(1, 1, 1, 1)
    out, S = o.recurrent(q, k, v, np.array([0.5]), state=S0)
    assert S.ravel()[0] == 0.5 * 2.0 + 3.0 * -1.0      # -2
    assert out.ravel()[0] == 4.0 * (0.5 * 2.0 - 3.0)   # -8
    out_c, S_c = o.chunkwise(q, k, v, np.array([0.5]), 1, state_in=S0)
    assert out_c.ravel()[0] == -8.0 and S_c.ravel()[0] == -2.0


# --- closed forms ------------------------------------------------------------

def check_closed_form_ones(o):
    """q = k = 1 (length dk), v = 1: o_n = sqrt(dk) (1-g^(n+1))/(1-g), S = (1-g^N)/(1-g)."""
    for dk, dv, N, g in ((4, 3, 37, 0.9), (9, 2, 20, 0.96875), (16, 5, 64, 0.5)):
        q = np.ones((1, 1, N, dk))
        k = np.ones((1, 1, N, dk))
        v = np.ones((1, 1, N, dv))
        n = np.arange(N, dtype=np.float64)
        want = (math.sqrt(dk) * (1.0 - g ** (n + 1)) / (1.0 - g))[:, None] * np.ones(dv)
        want_s = (1.0 - g ** N) / (1.0 - g) * np.ones((dk, dv))
        res = _all_forms(o, q, k, v, np.array([g]), chunks=(1, 5, 16, N))
        for name, (out, S) in res.items():
            _close(out[0, 0], want, 1e-13, f"ones {name}")
            if S is not None:
                _close(S[0, 0], want_s, 1e-13, f"ones state {name}")
        rows = o.parallel_rows(q[0, 0], k[0, 0], v[0, 0], g, [0, N // 2, N - 1])
        _close(rows, want[[0, N // 2, N - 1]], 1e-13, "ones rows")


def check_impulse(o):
    """One non-zero key/value at m0: o_n = g^(n-m0) (q_n.k_m0/sqrt(dk)) v_m0, n >= m0; 0 before."""
    N, dk, dv, m0, g = 24, 3, 4, 7, 0.8
    q = _rand((1, 1, N, dk), 1)
    k = np.zeros((1, 1, N, dk))
    v = np.zeros((1, 1, N, dv))
    k[0, 0, m0] = _rand(dk, 2)
    v[0, 0, m0] = _rand(dv, 3)
    want = np.zeros((N, dv))
    for n in range(m0, N):
        want[n] = g ** (n - m0) * (q[0, 0, n] @ k[0, 0, m0]) / math.sqrt(dk) * v[0, 0, m0]
    want_s = g ** (N - 1 - m0) * np.outer(k[0, 0, m0], v[0, 0, m0])
    res = _all_forms(o, q, k, v, np.array([g]), chunks=(1, 4, 5, N))
    for name, (out, S) in res.items():
        _close(out[0, 0], want, 1e-14, f"impulse {name}")
        assert np.all(out[0, 0, :m0] == 0.0), f"impulse {name}: output before the impulse"
        if S is not None:
            _close(S[0, 0], want_s, 1e-14, f"impulse state {name}")
    rows = o.parallel_rows(q[0, 0], k[0, 0], v[0, 0], g, [0, m0, N - 1])
    _close(rows, want[[0, m0, N - 1]], 1e-14, "impulse rows")


# --- special cases reducing to library routines --------------------------------

def check_gamma_one_is_causal_linear_attention(o):
    """gamma = 1: causal linear attention without normaliser, tril(QK^T)V/sqrt(dk)."""
    B, H, N, dk, dv = 2, 2, 29, 6, 5
    q, k, v = _rand((B, H, N, dk), 4), _rand((B, H, N, dk), 5), _rand((B, H, N, dv), 6)
    want = np.tril(q @ np.swapaxes(k, -1, -2)) @ v / math.sqrt(dk)
    want_s = np.swapaxes(k, -1, -2) @ v
    res = _all_forms(o, q, k, v, np.ones(H), chunks=(1, 7, N))
    for name, (out, S) in res.items():
        _close(out, want, 1e-13, f"gamma=1 {name}")
        if S is not None:
            _close(S, want_s, 1e-13, f"gamma=1 state {name}")


def check_gamma_zero_is_diagonal(o):
    """gamma = 0: D = I, o_n = (q_n.k_n/sqrt(dk)) v_n and S = k_{N-1}^T v_{N-1}."""
    B, H, N, dk, dv = 1, 2, 17, 4, 3
    q, k, v = _rand((B, H, N, dk), 7), _rand((B, H, N, dk), 8), _rand((B, H, N, dv), 9)
    want = np.sum(q * k, axis=-1, keepdims=True) / math.sqrt(dk) * v
    want_s = k[:, :, -1, :, None] * v[:, :, -1, None, :]
    res = _all_forms(o, q, k, v, np.zeros(H), chunks=(1, 4, N))
    for name, (out, S) in res.items():
        _close(out, want, 1e-14, f"gamma=0 {name}")
        if S is not None:
            _close(S, want_s, 1e-14, f"gamma=0 state {name}")


# --- the pages' invariant and structural properties ---------------------------

def check_three_forms_equal(o):
    """Parallel == recurrent == chunkwise, for every chunk size, ragged tails included."""
    B, H, dk, dv = 2, 3, 8, 6
    g = o.gamma(np.arange(H))
    for N in (1, 16, 45):
        q, k, v = (_rand((B, H, N, dk), 10 + N), _rand((B, H, N, dk), 11 + N),
                   _rand((B, H, N, dv), 12 + N))
        res = _all_forms(o, q, k, v, g, chunks=(1, 2, 3, 7, 16, N, N + 5))
        ref_out, ref_s = res["recurrent"]
        for name, (out, S) in res.items():
            _close(out, ref_out, 1e-12, f"N={N} {name} vs recurrent")
            if S is not None:
                _close(S, ref_s, 1e-12, f"N={N} {name} state vs recurrent")
        for b, h in ((0, 0), (1, 2)):
            rows = [0, N // 2, N - 1]
            got = o.parallel_rows(q[b, h], k[b, h], v[b, h], g[h], rows)
            _close(got, ref_out[b, h, rows], 1e-12, f"N={N} rows ({b},{h})")


def check_linearity_and_heads(o):
    """Output is linear in V and in Q; permuting heads with their gammas permutes outputs."""
    B, H, N, dk, dv = 1, 4, 21, 5, 4
    q, k = _rand((B, H, N, dk), 20), _rand((B, H, N, dk), 21)
    v1, v2 = _rand((B, H, N, dv), 22), _rand((B, H, N, dv), 23)
    g = np.array([0.9, 0.5, 0.99, 0.7])
    o1, _ = o.chunkwise(q, k, v1, g, 4)
    o2, _ = o.chunkwise(q, k, v2, g, 4)
    o12, _ = o.chunkwise(q, k, 2.0 * v1 - 3.0 * v2, g, 4)
    _close(o12, 2.0 * o1 - 3.0 * o2, 1e-13, "linear in V")
    q2 = _rand((B, H, N, dk), 24)
    oq, _ = o.chunkwise(q2, k, v1, g, 4)
    oqq, _ = o.chunkwise(q + q2, k, v1, g, 4)
    _close(oqq, o1 + oq, 1e-13, "linear in Q")
    perm = np.array([2, 0, 3, 1])
    op, Sp = o.chunkwise(q[:, perm], k[:, perm], v1[:, perm], g[perm], 4)
    _, S1 = o.chunkwise(q, k, v1, g, 4)
    _close(op, o1[:, perm], 1e-15, "head permutation")
    _close(Sp, S1[:, perm], 1e-15, "head permutation state")


def check_state_continuation(o):
    """The state summarises the past: prefix state + recurrent/chunkwise on the rest == whole."""
    B, H, N, dk, dv, cut = 1, 2, 40, 6, 7, 23
    g = np.array([0.95, 0.8])
    q, k, v = _rand((B, H, N, dk), 30), _rand((B, H, N, dk), 31), _rand((B, H, N, dv), 32)
    full_o, full_s = o.chunkwise(q, k, v, g, 8)
    pre_o, pre_s = o.chunkwise(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut], g, 8)
    rest_o, rest_s = o.recurrent(q[:, :, cut:], k[:, :, cut:], v[:, :, cut:], g, state=pre_s)
    _close(pre_o, full_o[:, :, :cut], 1e-13, "prefix")
    _close(rest_o, full_o[:, :, cut:], 1e-13, "continuation (recurrent)")
    _close(rest_s, full_s, 1e-13, "continuation state (recurrent)")
    rest_o2, rest_s2 = o.chunkwise(q[:, :, cut:], k[:, :, cut:], v[:, :, cut:], g, 5,
                                   state_in=pre_s)
    _close(rest_o2, full_o[:, :, cut:], 1e-13, "continuation (chunkwise)")
    _close(rest_s2, full_s, 1e-13, "continuation state (chunkwise)")


def check_empty_sequence(o):
    """N = 0: no outputs; the final state is the starting state (zero by default)."""
    q = np.zeros((1, 2, 0, 4))
    v = np.zeros((1, 2, 0, 3))
    out, S = o.chunkwise(q, q, v, np.array([0.9, 0.5]), 4)
    assert out.shape == (1, 2, 0, 3) and np.all(S == 0.0)
    S0 = _rand((1, 2, 4, 3), 40)
    _, S2 = o.recurrent(q, q, v, np.array([0.9, 0.5]), state=S0)
    assert np.array_equal(S2, S0)


# --- the normalisation of the heads' outputs -----------------------------------

def check_groupnorm_is_the_library_group_norm(o):
    """Per-(token, head) normalisation == torch.nn.functional.group_norm with
    one group per head over the concatenated head channels (fp64, CPU), with a
    random affine and two values of eps (the large one would expose eps
    applied outside the square root)."""
    import torch
    B, H, N, dv = 2, 3, 7, 12
    r = _rand((B, H, N, dv), 50) * 3.0 + 0.5
    w, bias = _rand((H * dv,), 51), _rand((H * dv,), 52)
    for eps in (1e-6, 0.5):
        y = o.groupnorm(r, w, bias, eps)
        x = torch.from_numpy(np.ascontiguousarray(r.transpose(0, 2, 1, 3))).reshape(B * N, H * dv)
        ref = torch.nn.functional.group_norm(x, H, torch.from_numpy(w), torch.from_numpy(bias), eps)
        _close(y, ref.reshape(B, N, H, dv).numpy(), 1e-13, f"groupnorm vs library, eps {eps}")


def check_groupnorm_invariants(o):
    """Constant groups give the bias; without an affine every group has mean 0
    and mean square var/(var+eps); with eps = 0 the result ignores a positive
    scale and a shift of each group; permuting heads permutes the output's head
    axis."""
    B, H, N, dv = 1, 2, 5, 8
    bias = _rand((H * dv,), 60)
    const = np.broadcast_to(_rand((B, H, N, 1), 61), (B, H, N, dv)).copy()
    y = o.groupnorm(const, _rand((H * dv,), 62), bias, 1e-6)
    # (x - mu is a rounding error of the mean, magnified by 1/sqrt(eps))
    _close(y, np.broadcast_to(bias.reshape(1, 1, H, dv), y.shape), 1e-10, "groupnorm of constants")
    r = _rand((B, H, N, dv), 63)
    y = o.groupnorm(r, None, None, 1e-6)
    var = r.var(axis=-1).transpose(0, 2, 1)
    assert np.max(np.abs(y.mean(axis=-1))) < 1e-14
    _close((y ** 2).mean(axis=-1), var / (var + 1e-6), 1e-13, "groupnorm mean square")
    _close(o.groupnorm(7.5 * r - 2.0, None, None, 0.0), o.groupnorm(r, None, None, 0.0), 1e-12,
           "groupnorm scale and shift")
    yp = o.groupnorm(r[:, ::-1].copy(), None, None, 1e-6)
    _close(yp, y[:, :, ::-1], 0.0, "groupnorm head permutation")


# --- the position phase rotation -------------------------------------------------

def check_rotation_relative_position(o):
    """Rotated query and key give scores that depend on n - m only (a shift of
    both positions leaves every score unchanged), and equal the unrotated pair
    with the key turned by (m - n) theta."""
    d, N = 8, 9
    th = np.abs(_rand((d // 2,), 70))
    q, k = _rand((1, 1, N, d), 71), _rand((1, 1, N, d), 72)
    s0 = o.rotate(q, th, 0)[0, 0] @ o.rotate(k, th, 0)[0, 0].T
    s5 = o.rotate(q, th, 5)[0, 0] @ o.rotate(k, th, 5)[0, 0].T
    _close(s5, s0, 1e-12, "rotation: shift invariance")
    n, m = 6, 2
    k_rel = o.rotate(k[:, :, m:m + 1], th, m - n)  # key turned by (m - n) theta
    want = q[0, 0, n] @ k_rel[0, 0, 0]
    _close(s0[n, m], want, 1e-12, "rotation: relative angle")


def check_rotation_special_cases(o):
    """Position 0 and theta = 0 are the identity; lengths of pairs are kept;
    a quarter turn maps (1, 0) to (0, 1); rotations compose."""
    x = _rand((2, 3, 4, 6), 73)
    th = np.abs(_rand((3,), 74))
    y = o.rotate(x, th, 0)
    assert np.array_equal(y[:, :, 0], x[:, :, 0])
    assert np.array_equal(o.rotate(x, np.zeros(3), 7), x)
    _close(np.hypot(y[..., 0::2], y[..., 1::2]), np.hypot(x[..., 0::2], x[..., 1::2]), 1e-14,
           "rotation keeps pair lengths")
    e = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    _close(o.rotate(e, np.array([np.pi / 2]), 1), np.array([0.0, 1.0]).reshape(1, 1, 1, 2), 1e-15,
           "quarter turn")
    x1 = x[:, :, :1]
    _close(o.rotate(o.rotate(x1, th, 3), th, 4), o.rotate(x1, th, 7), 1e-13, "rotations compose")


# --- the backward pass -------------------------------------------------------------

def _loss(o, q, k, v, g, dout, dstate, state_in):
    """sum(dout * out) + sum(dstate * S_N) for the forward from state_in."""
    out, S = o.recurrent(q, k, v, g, state=state_in)
    return float(np.sum(dout * out) + (0.0 if dstate is None else np.sum(dstate * S)))


def check_backward_hand_expanded(o):
    gold = _read_golden("backward_hand_n2.txt")
    sh = (1, 1, 2, 1)
    q, k, v, dout = (gold[x].reshape(sh) for x in ("q", "k", "v", "dout"))
    S0, dS = gold["state_in"].reshape(1, 1, 1, 1), gold["dstate"].reshape(1, 1, 1, 1)
    dq, dk, dv, ds0 = o.backward(q, k, v, gold["gamma"], dout, dS, S0)
    assert np.array_equal(dq.ravel(), gold["dq"]), dq.ravel()
    assert np.array_equal(dk.ravel(), gold["dk"]), dk.ravel()
    assert np.array_equal(dv.ravel(), gold["dv"]), dv.ravel()
    assert np.array_equal(ds0.ravel(), gold["dstate_in"]), ds0.ravel()


def check_backward_is_the_derivative(o):
    """The forward is linear in each of q, k, v and the starting state, so
    L(x + e) - L(x) equals <dL/dx, e> exactly up to rounding for any e: checked
    for random directions, with and without a starting state and a final-state
    gradient, for decays 0.9, 0.5, 0 and 1."""
    B, H, N, dk, dv = 2, 4, 13, 5, 3
    g = np.array([0.9, 0.5, 0.0, 1.0])
    q, k, v = _rand((B, H, N, dk), 80), _rand((B, H, N, dk), 81), _rand((B, H, N, dv), 82)
    dout, S0, dS = _rand((B, H, N, dv), 83), _rand((B, H, dk, dv), 84), _rand((B, H, dk, dv), 85)
    for s0, ds in ((S0, dS), (None, None), (S0, None), (None, dS)):
        grads = o.backward(q, k, v, g, dout, ds, s0)
        base = _loss(o, q, k, v, g, dout, ds, s0)
        args = [q, k, v, np.zeros((B, H, dk, dv)) if s0 is None else s0]
        for which, grad in enumerate(grads):
            e = _rand(args[which].shape, 90 + which)
            moved = list(args)
            moved[which] = args[which] + e
            got = _loss(o, *moved[:3], g, dout, ds, moved[3]) - base
            want = float(np.sum(grad * e))
            assert abs(got - want) <= 1e-11 * max(1.0, abs(want)), (which, got, want)


def check_backward_brute_force_tiny(o):
    """Every entry of every gradient, one unit direction at a time (N = 3,
    d_k = d_v = 2, starting state and final-state gradient present)."""
    B, H, N, dk, dv = 1, 1, 3, 2, 2
    g = np.array([0.75])
    q, k, v = _rand((B, H, N, dk), 86), _rand((B, H, N, dk), 87), _rand((B, H, N, dv), 88)
    dout, S0, dS = _rand((B, H, N, dv), 89), _rand((B, H, dk, dv), 90), _rand((B, H, dk, dv), 91)
    grads = o.backward(q, k, v, g, dout, dS, S0)
    base = _loss(o, q, k, v, g, dout, dS, S0)
    args = [q, k, v, S0]
    for which, grad in enumerate(grads):
        for idx in np.ndindex(*args[which].shape):
            moved = [a.copy() for a in args]
            moved[which][idx] += 1.0
            got = _loss(o, *moved[:3], g, dout, dS, moved[3]) - base
            assert abs(got - grad[idx]) <= 1e-12 * max(1.0, abs(got)), (which, idx, got, grad[idx])


def check_backward_euler_identities(o):
    """out is linear in q, and out and S_N are jointly linear in (k, S0) and in
    (v, S0), so <dq, q> = <dout, out> and <dk, k> + <dS0, S0> = <dv, v> +
    <dS0, S0> = L; these hold at any size."""
    B, H, N, dk, dv = 1, 3, 40, 8, 6
    g = np.array([0.96875, 0.7, 0.2])
    q, k, v = _rand((B, H, N, dk), 92), _rand((B, H, N, dk), 93), _rand((B, H, N, dv), 94)
    dout, S0, dS = _rand((B, H, N, dv), 95), _rand((B, H, dk, dv), 96), _rand((B, H, dk, dv), 97)
    out, S = o.recurrent(q, k, v, g, state=S0)
    dq, dk_, dv_, ds0 = o.backward(q, k, v, g, dout, dS, S0)
    lo, L = np.sum(dout * out), np.sum(dout * out) + np.sum(dS * S)
    _close(np.sum(dq * q), lo, 1e-13, "<dq, q>")
    _close(np.sum(dk_ * k) + np.sum(ds0 * S0), L, 1e-13, "<dk, k> + <dS0, S0>")
    _close(np.sum(dv_ * v) + np.sum(ds0 * S0), L, 1e-13, "<dv, v> + <dS0, S0>")


def check_backward_gamma_one_is_library_autograd(o):
    """With gamma = 1 and no states the forward is tril(Q K^T) V / sqrt(d_k), so
    its gradients are those torch's autograd gives for that product (fp64)."""
    import torch
    B, H, N, dk, dv = 1, 2, 17, 4, 3
    q, k, v = _rand((B, H, N, dk), 98), _rand((B, H, N, dk), 99), _rand((B, H, N, dv), 100)
    dout = _rand((B, H, N, dv), 101)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    out = torch.tril(tq @ tk.transpose(-1, -2)) @ tv / math.sqrt(dk)
    out.backward(torch.from_numpy(dout))
    dq, dk_, dv_, ds0 = o.backward(q, k, v, np.ones(H), dout)
    _close(dq, tq.grad.numpy(), 1e-13, "dq vs autograd")
    _close(dk_, tk.grad.numpy(), 1e-13, "dk vs autograd")
    _close(dv_, tv.grad.numpy(), 1e-13, "dv vs autograd")
    want_ds0 = np.einsum("bhnk,bhnv->bhkv", q, dout) / math.sqrt(dk)
    _close(ds0, want_ds0, 1e-13, "dS0 at gamma = 1")


def check_backward_scans_are_forward_retentions(o):
    """Each gradient is a retention forward of permuted operands (decays > 0):
    dq is the chunkwise form of (dout, v, k) from S0^T, times sqrt(dv)/sqrt(dk)
    (that forward divides by the square root of its query width, dv); dv is
    the time-reversed form of (k, q, dout) from dS/(s g); dk is the
    time-reversed form of (v, dout, q) from dS^T/(s g), times s sqrt(dv); and
    dS0 is s g times the final state of the reversed dv form (s = 1/sqrt(dk))."""
    B, H, N, dk, dv = 1, 4, 37, 6, 10
    g = np.array([0.9, 0.5, 0.99, 1.0])  # 1.0: no decay at all, the edge of the schedule
    q, k = _rand((B, H, N, dk), 103), _rand((B, H, N, dk), 104)
    v, dout = _rand((B, H, N, dv), 105), _rand((B, H, N, dv), 106)
    S0, dS = _rand((B, H, dk, dv), 107), _rand((B, H, dk, dv), 108)
    dq, dk_, dv_, ds0 = o.backward(q, k, v, g, dout, dS, S0)
    s = 1.0 / math.sqrt(dk)
    gs = g[None, :, None, None]
    T = lambda x: np.ascontiguousarray(x.transpose(0, 1, 3, 2))
    rev = lambda x: np.ascontiguousarray(x[:, :, ::-1])
    fq, _ = o.chunkwise(dout, v, k, g, 8, state_in=T(S0))
    _close(dq, fq * math.sqrt(dv) / math.sqrt(dk), 1e-13, "dq as a forward")
    fv, sv = o.chunkwise(rev(k), rev(q), rev(dout), g, 8, state_in=dS / (s * gs))
    _close(dv_, rev(fv), 1e-13, "dv as a reversed forward")
    _close(ds0, s * gs * sv, 1e-13, "dS0 as the reversed forward's state")
    fk, _ = o.chunkwise(rev(v), rev(dout), rev(q), g, 8, state_in=T(dS) / (s * gs))
    _close(dk_, rev(fk) * math.sqrt(dv) * s, 1e-13, "dk as a reversed forward")

def check_backward_zero_decay_as_forwards(o):
    """Decay 0, where the division by s g of the previous pin does not exist:
    dq is still the forward of (dout, v, k) from S0^T; dv and dk are the
    reversed forwards from a zero state, and the final-state gradient reaches
    the last token alone (0^0 = 1, every other power of 0 vanishes):
    dv_{N-1} += k_{N-1} dS, dk_{N-1} += v_{N-1} dS^T, and dS0 = 0 when N > 0.
    A second head with decay 0.7 runs beside it in the same calls."""
    B, H, N, dk, dv = 2, 2, 19, 4, 6
    g = np.array([0.0, 0.7])
    q, k = _rand((B, H, N, dk), 113), _rand((B, H, N, dk), 114)
    v, dout = _rand((B, H, N, dv), 115), _rand((B, H, N, dv), 116)
    S0, dS = _rand((B, H, dk, dv), 117), _rand((B, H, dk, dv), 118)
    dq, dk_, dv_, ds0 = o.backward(q, k, v, g, dout, dS, S0)
    s = 1.0 / math.sqrt(dk)
    T = lambda x: np.ascontiguousarray(x.transpose(0, 1, 3, 2))
    rev = lambda x: np.ascontiguousarray(x[:, :, ::-1])
    fq, _ = o.chunkwise(dout, v, k, g, 5, state_in=T(S0))
    _close(dq[:, :1], (fq * math.sqrt(dv) / math.sqrt(dk))[:, :1], 1e-13, "dq as a forward, decay 0")
    fv, _ = o.chunkwise(rev(k), rev(q), rev(dout), g, 5)
    want_dv = rev(fv)[:, :1].copy()
    want_dv[:, 0, N - 1] += np.einsum("bi,bij->bj", k[:, 0, N - 1], dS[:, 0])
    _close(dv_[:, :1], want_dv, 1e-13, "dv as a reversed forward plus the last token's dS term, decay 0")
    fk, _ = o.chunkwise(rev(v), rev(dout), rev(q), g, 5)
    want_dk = (rev(fk) * math.sqrt(dv) * s)[:, :1].copy()
    want_dk[:, 0, N - 1] += np.einsum("bj,bij->bi", v[:, 0, N - 1], dS[:, 0])
    _close(dk_[:, :1], want_dk, 1e-13, "dk as a reversed forward plus the last token's dS term, decay 0")
    assert np.array_equal(ds0[:, 0], np.zeros_like(ds0[:, 0])), "dS0 must vanish at decay 0"


def check_backward_empty_sequence(o):
    """N = 0: no gradients of the sequence; the starting state's gradient is dS."""
    q = np.zeros((1, 2, 0, 4))
    v = np.zeros((1, 2, 0, 3))
    dS = _rand((1, 2, 4, 3), 102)
    dq, dk, dv, ds0 = o.backward(q, q, v, np.array([0.9, 0.0]), v, dS)
    assert dq.shape == (1, 2, 0, 4) and dv.shape == (1, 2, 0, 3)
    assert np.array_equal(ds0, dS)


ALL_CHECKS = [
    check_gamma_printed,
    check_hand_expanded_scalar,
    check_hand_expanded_vector,
    check_one_step_from_state,
    check_closed_form_ones,
    check_impulse,
    check_gamma_one_is_causal_linear_attention,
    check_gamma_zero_is_diagonal,
    check_three_forms_equal,
    check_linearity_and_heads,
    check_state_continuation,
    check_empty_sequence,
    check_groupnorm_is_the_library_group_norm,
    check_groupnorm_invariants,
    check_rotation_relative_position,
    check_rotation_special_cases,
    check_backward_hand_expanded,
    check_backward_is_the_derivative,
    check_backward_brute_force_tiny,
    check_backward_euler_identities,
    check_backward_gamma_one_is_library_autograd,
    check_backward_scans_are_forward_retentions,
    check_backward_zero_decay_as_forwards,
    check_backward_empty_sequence,
]
