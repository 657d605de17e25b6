"""Pins of the fp64 oracle against facts that the pages and the mathematics fix (CPU only).

None of these re-types the oracle's formulas. The checks are:
  * finite differences of the scalar loss sum(dy * out), over every input element (tiny shapes);
  * symbolic differentiation of the forward definition (sympy; an independent derivation of BPTT);
  * the closed-form geometric series for constant delta, u, B, C (forward);
  * the delta == 0 special case. It reduces to the inclusive reverse running sum of
    cumsum_backward_row (rlx-cpu src/training_bwd.rs). A hand-worked integer fixture covers it.
  * T == 1, where every gradient is a hand-computable product;
  * the Euler identities: out is homogeneous of degree 1 in u, in B, in C and in D;
  * the SiLU-gradient identity sigma*(1 + x*(1 - sigma)) == sigma*(1 - silu) + silu.
    The first form is from mamba-rs src/mamba_ssm/cpu/backward.rs, Phase B2; the second from
    luma-tensor src/grad/backprop.rs, UnaryOp::Silu.
Planted mistakes also go in: edited copies of the oracle source, each of which must fail at
least one pin.
"""
import os

import numpy as np
import pytest

import oracle
import synth

GRAD_KEYS = ("d_delta", "d_u", "d_B", "d_C", "d_gate", "d_A_log", "d_D")
INPUT_OF = {"d_delta": "delta", "d_u": "u", "d_B": "B", "d_C": "C", "d_gate": "gate",
            "d_A_log": "A_log", "d_D": "D"}


def _tiny_random(seed=3, batch=2, T=5, Di=3, N=4):
    x = oracle.as64(synth.random_inputs(batch, T, Di, N, seed=seed, a_log_random=True))
    return x


def fd_max_rel_err(x, lib=None, per_tensor=None, seed=0):
    """max over tensors of max|fd - analytic| / max(1, max|analytic|)."""
    g = oracle.bwd(x, lib=lib)
    rng = np.random.default_rng(seed)
    worst = 0.0
    for gk in GRAD_KEYS:
        xk = INPUT_OF[gk]
        flat = x[xk].reshape(-1)
        idx = np.arange(flat.size)
        if per_tensor is not None and flat.size > per_tensor:
            idx = rng.choice(flat.size, per_tensor, replace=False)
        an = g[gk].reshape(-1)
        scale = max(1.0, float(np.abs(an).max()))
        for i in idx:
            orig = flat[i]
            h = 1e-6 * max(1.0, abs(orig))
            flat[i] = orig + h
            lp = oracle.loss(x, lib=lib)
            flat[i] = orig - h
            lm = oracle.loss(x, lib=lib)
            flat[i] = orig
            fd = (lp - lm) / (2 * h)
            worst = max(worst, abs(fd - an[i]) / scale)
    return worst


def geo_max_rel_err(lib=None):
    """Constant delta, u, B, C over t: h_t[n] = delta*u*B[n] * (1 - a^(t+1)) / (1 - a)."""
    batch, T, Di, N = 2, 40, 3, 5
    rng = np.random.default_rng(11)
    dl = rng.uniform(0.05, 0.6, size=(batch, Di))
    uu = rng.normal(size=(batch, Di))
    Bn = rng.normal(size=(batch, N))
    Cn = rng.normal(size=(batch, N))
    A_log = rng.uniform(-1, 1, size=(Di, N))
    D = rng.uniform(0.5, 1.5, size=Di)
    gate = rng.normal(size=(batch, T, Di))
    x = {"delta": np.repeat(dl[:, None, :], T, 1), "u": np.repeat(uu[:, None, :], T, 1),
         "B": np.repeat(Bn[:, None, :], T, 1), "C": np.repeat(Cn[:, None, :], T, 1),
         "gate": gate, "A_log": A_log, "D": D, "dy": np.zeros((batch, T, Di))}
    x = oracle.as64(x)
    out, y = oracle.fwd(x, lib=lib)
    A = -np.exp(A_log)                                   # [Di, N]
    a = np.exp(dl[:, :, None] * A[None])                 # [batch, Di, N]
    t = np.arange(T)[None, :, None, None]
    h = (dl * uu)[:, None, :, None] * Bn[:, None, None, :] * (1 - a[:, None] ** (t + 1)) / (1 - a[:, None])
    y_ref = np.einsum("btdn,bn->btd", h, Cn) + D[None, None, :] * uu[:, None, :]
    sig = 1 / (1 + np.exp(-gate))
    out_ref = y_ref * gate * sig
    return max(float(np.abs(y - y_ref).max() / np.abs(y_ref).max()),
               float(np.abs(out - out_ref).max() / np.abs(out_ref).max()))


def delta_zero_max_err(lib=None):
    """delta == 0: h == 0, y = D*u, d_B = d_C = d_A_log = 0, d_u = d_y*D and
    d_delta_t = u_t * sum_n B_t[n] * S_t[n] with S the inclusive reverse running sum of d_y*C."""
    batch, T, Di, N = 2, 30, 4, 3
    x = oracle.as64(synth.random_inputs(batch, T, Di, N, seed=5, a_log_random=True))
    x["delta"][:] = 0.0
    g = oracle.bwd(x, lib=lib)
    out, y = oracle.fwd(x, lib=lib)
    sig = 1 / (1 + np.exp(-x["gate"]))
    d_y = x["dy"] * x["gate"] * sig                                  # [b,T,Di]
    contrib = d_y[..., None] * x["C"][:, :, None, :]                 # [b,T,Di,N]
    S = np.empty_like(contrib)
    run = np.zeros_like(contrib[:, 0])
    for t in range(T - 1, -1, -1):                                   # inclusive suffix sum
        run = run + contrib[:, t]
        S[:, t] = run
    dd_ref = x["u"] * np.einsum("btdn,btn->btd", S, x["B"])
    errs = [np.abs(y - x["D"] * x["u"]).max(),
            np.abs(g["d_B"]).max(), np.abs(g["d_C"]).max(), np.abs(g["d_A_log"]).max(),
            np.abs(g["d_u"] - d_y * x["D"]).max() / max(1.0, np.abs(d_y * x["D"]).max()),
            np.abs(g["d_delta"] - dd_ref).max() / np.abs(dd_ref).max()]
    return float(max(errs))


def t1_max_err(lib=None):
    """T == 1: h = delta*u*B; every gradient is a closed-form product."""
    batch, T, Di, N = 3, 1, 4, 5
    x = oracle.as64(synth.random_inputs(batch, T, Di, N, seed=7, a_log_random=True))
    g = oracle.bwd(x, lib=lib)
    out, y = oracle.fwd(x, lib=lib)
    dl, uu, gt, dy = (x[k][:, 0] for k in ("delta", "u", "gate", "dy"))   # [b, Di]
    Bn, Cn = x["B"][:, 0], x["C"][:, 0]                                   # [b, N]
    CB = np.sum(Cn * Bn, axis=1)[:, None]                                 # [b, 1]
    s = 1 / (1 + np.exp(-gt))
    y_ref = dl * uu * CB + x["D"] * uu
    d_y = dy * gt * s
    ref = {
        "out": y_ref * gt * s,
        "d_delta": d_y * uu * CB,
        "d_u": d_y * (dl * CB + x["D"]),
        "d_gate": dy * y_ref * s * (1 + gt * (1 - s)),
        "d_B": np.einsum("bd,bn->bn", d_y * dl * uu, Cn),
        "d_C": np.einsum("bd,bn->bn", d_y * dl * uu, Bn),
        "d_D": np.sum(d_y * uu, axis=0),
        "d_A_log": np.zeros_like(x["A_log"]),
    }
    got = {"out": out[:, 0], "d_delta": g["d_delta"][:, 0], "d_u": g["d_u"][:, 0],
           "d_gate": g["d_gate"][:, 0], "d_B": g["d_B"][:, 0], "d_C": g["d_C"][:, 0],
           "d_D": g["d_D"], "d_A_log": g["d_A_log"]}
    return max(float(np.abs(got[k] - ref[k]).max() / max(1.0, np.abs(ref[k]).max())) for k in ref)


def euler_max_err(lib=None):
    x = oracle.as64(synth.random_inputs(2, 50, 8, 6, seed=9, a_log_random=True))
    g = oracle.bwd(x, lib=lib)
    out, y = oracle.fwd(x, lib=lib)
    s = 1 / (1 + np.exp(-x["gate"]))
    w = x["dy"] * x["gate"] * s                         # dL/dy
    lhs_rhs = [
        (np.sum(g["d_u"] * x["u"]), np.sum(x["dy"] * out)),
        (np.sum(g["d_B"] * x["B"]), np.sum(w * (y - x["D"] * x["u"]))),
        (np.sum(g["d_C"] * x["C"]), np.sum(w * (y - x["D"] * x["u"]))),
        (np.sum(g["d_D"] * x["D"]), np.sum(w * x["D"] * x["u"])),
    ]
    return max(abs(a - b) / max(1.0, abs(b)) for a, b in lhs_rhs)


def softplus_chain_fd_max_rel_err(lib=None):
    """The softplus variant end to end: with delta = softplus(raw), finite differences of the
    loss over every raw element against softplus_bwd(raw, d_delta). Raw values straddle the
    threshold 20 (the identity branch) and large negative values."""
    x = _tiny_random(seed=7)
    rng = np.random.default_rng(7)
    raw = rng.normal(-1.0, 2.0, size=x["delta"].shape)
    raw.reshape(-1)[:3] = [24.0, 20.5, -25.0]
    x["delta_raw"] = raw
    d_delta = oracle.bwd(oracle.with_softplus(x, lib), lib=lib)["d_delta"]
    an = oracle.softplus_bwd(raw, d_delta, lib).reshape(-1)
    scale = max(1.0, float(np.abs(an).max()))
    flat = raw.reshape(-1)
    worst = 0.0
    for i in range(flat.size):
        orig = flat[i]
        h = 1e-6 * max(1.0, abs(orig))
        flat[i] = orig + h
        lp = oracle.loss(oracle.with_softplus(x, lib), lib=lib)
        flat[i] = orig - h
        lm = oracle.loss(oracle.with_softplus(x, lib), lib=lib)
        flat[i] = orig
        worst = max(worst, abs((lp - lm) / (2 * h) - an[i]) / scale)
    return worst


def softplus_identity_max_err(lib=None):
    """softplus(x) - softplus(-x) = x for |x| <= 20 (log(1 + e^x) - log(1 + e^-x) = x), and the
    identity branch above 20: softplus(x) = x and d_raw = d_delta exactly."""
    x = np.linspace(-20.0, 20.0, 401)
    e1 = float(np.abs(oracle.softplus(x, lib) - oracle.softplus(-x, lib) - x).max())
    hi = np.array([20.0 + 1e-9, 25.0, 80.0])
    g = np.array([0.3, -1.5, 2.0])
    e2 = float(np.abs(oracle.softplus(hi, lib) - hi).max())
    e3 = float(np.abs(oracle.softplus_bwd(hi, g, lib) - g).max())
    return max(e1, e2, e3)


def conv_fd_max_rel_err(lib=None, K=4, shape=(2, 9, 3), seed=11):
    """Causal conv1d + SiLU: finite differences of sum(d_u * u) over every element of x, w and
    bias against the oracle's backward (Phase B6 with its shift-register carry)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape)
    w = rng.standard_normal((shape[2], K)) * 0.7
    bias = rng.standard_normal(shape[2]) * 0.3
    d_u = rng.standard_normal(shape)
    g = oracle.conv_bwd(x, w, bias, d_u, lib)

    def loss():
        return float(np.sum(d_u * oracle.conv_fwd(x, w, bias, lib)[0]))
    worst = 0.0
    for arr, key in ((x, "d_x"), (w, "d_w"), (bias, "d_bias")):
        an = g[key].reshape(-1)
        scale = max(1.0, float(np.abs(an).max()))
        flat = arr.reshape(-1)
        for i in range(flat.size):
            orig = flat[i]
            h = 1e-6 * max(1.0, abs(orig))
            flat[i] = orig + h
            lp = loss()
            flat[i] = orig - h
            lm = loss()
            flat[i] = orig
            worst = max(worst, abs((lp - lm) / (2 * h) - an[i]) / scale)
    return worst


def conv_impulse_max_err(lib=None, K=4):
    """A unit impulse at step t0 with zero bias: pre[t0 + m] = w[d, K-1-m] for m < K and 0
    elsewhere (a causal filter's impulse response); u = pre * sigmoid(pre)."""
    T, Di, t0 = 10, 2, 3
    w = np.arange(1, Di * K + 1, dtype=np.float64).reshape(Di, K) / 7.0
    x = np.zeros((1, T, Di))
    x[0, t0, :] = 1.0
    u, pre = oracle.conv_fwd(x, w, np.zeros(Di), lib)
    want = np.zeros((T, Di))
    for m in range(K):
        want[t0 + m] = w[:, K - 1 - m]
    e1 = float(np.abs(pre[0] - want).max())
    e2 = float(np.abs(u[0] - want / (1.0 + np.exp(-want))).max())
    return max(e1, e2)


PINS = {
    "conv_fd": lambda lib: conv_fd_max_rel_err(lib) < 1e-6,
    "conv_fd_k2": lambda lib: conv_fd_max_rel_err(lib, K=2, shape=(1, 6, 2), seed=5) < 1e-6,
    "conv_impulse": lambda lib: conv_impulse_max_err(lib) < 1e-14,
    "softplus_fd": lambda lib: softplus_chain_fd_max_rel_err(lib) < 1e-6,
    "softplus_identity": lambda lib: softplus_identity_max_err(lib) < 1e-12,
    "fd": lambda lib: fd_max_rel_err(_tiny_random(), lib=lib) < 1e-6,
    "geo": lambda lib: geo_max_rel_err(lib) < 1e-12,
    "delta0": lambda lib: delta_zero_max_err(lib) < 1e-12,
    "t1": lambda lib: t1_max_err(lib) < 1e-12,
    "euler": lambda lib: euler_max_err(lib) < 1e-10,
}


# ----------------------------------------------------------------------------------------------
def test_fd_all_elements_tiny():
    assert fd_max_rel_err(_tiny_random()) < 1e-6


def test_fd_all_elements_odd_shape():
    assert fd_max_rel_err(_tiny_random(seed=4, batch=1, T=9, Di=2, N=3)) < 1e-6


def test_fd_sampled_tiny_workload():
    x = oracle.as64(synth.make_inputs(synth.BY_NAME["tiny"]))
    assert fd_max_rel_err(x, per_tensor=12, seed=1) < 1e-6


def test_softplus_chain_finite_differences():
    assert softplus_chain_fd_max_rel_err() < 1e-6


def test_softplus_identity_and_threshold():
    assert softplus_identity_max_err() < 1e-12
    # softplus(0) = ln 2 and softplus'(0) = 1/2 (values of the definition at zero)
    assert abs(oracle.softplus(np.array([0.0]))[0] - np.log(2.0)) < 1e-15
    assert oracle.softplus_bwd(np.array([0.0]), np.array([1.0]))[0] == 0.5


def test_conv_finite_differences():
    assert conv_fd_max_rel_err() < 1e-6
    assert conv_fd_max_rel_err(K=2, shape=(1, 6, 2), seed=5) < 1e-6
    assert conv_fd_max_rel_err(K=1, shape=(2, 5, 3), seed=6) < 1e-6


def test_conv_impulse_response():
    assert conv_impulse_max_err() < 1e-14
    assert conv_impulse_max_err(K=3) < 1e-14


def test_conv_kernel_size_one_is_pointwise():
    """K = 1: pre = w*x + b per element, so d_x = d_pre * w exactly as a product."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 4, 3))
    w = rng.standard_normal((3, 1))
    b = rng.standard_normal(3)
    du = rng.standard_normal((2, 4, 3))
    u, pre = oracle.conv_fwd(x, w, b)
    assert np.allclose(pre, x * w[:, 0] + b, rtol=0, atol=1e-14)
    g = oracle.conv_bwd(x, w, b, du)
    s = 1.0 / (1.0 + np.exp(-pre))
    dp = du * (s * (1 - pre * s) + pre * s)    # d/dp [p * sigmoid(p)], expanded differently
    assert np.allclose(g["d_x"], dp * w[:, 0], rtol=1e-12, atol=1e-14)
    assert np.allclose(g["d_bias"], dp.sum(axis=(0, 1)), rtol=1e-12, atol=1e-14)


def test_geometric_closed_form():
    assert geo_max_rel_err() < 1e-12


def test_delta_zero_reduces_to_suffix_sum():
    assert delta_zero_max_err() < 1e-12


def test_t1_closed_form():
    assert t1_max_err() < 1e-12


def test_euler_identities():
    assert euler_max_err() < 1e-10


def _read_golden(name):
    vals = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = np.array([float(t) for t in v])
    return vals


def test_golden_delta_zero_integer_example():
    g = _read_golden("delta_zero_suffix_sum.txt")
    b, T, Di, N = (int(g[k][0]) for k in ("batch", "T", "d_inner", "d_state"))
    x = {"delta": g["delta"].reshape(b, T, Di), "u": g["u"].reshape(b, T, Di),
         "B": g["B"].reshape(b, T, N), "C": g["C"].reshape(b, T, N),
         "gate": g["gate"].reshape(b, T, Di), "dy": g["dy"].reshape(b, T, Di),
         "A_log": g["A_log"].reshape(Di, N), "D": g["D"].reshape(Di)}
    x = oracle.as64(x)
    out, y = oracle.fwd(x)
    gr = oracle.bwd(x)
    np.testing.assert_array_equal(out.reshape(-1), g["expect_out"])
    np.testing.assert_array_equal(y.reshape(-1), g["expect_y"])
    for k in GRAD_KEYS:
        np.testing.assert_array_equal(gr[k].reshape(-1), g["expect_" + k], err_msg=k)


def test_silu_gradient_two_forms():
    """Phase B2's sigma*(1 + x*(1 - sigma)) equals luma-tensor's sigma*(1 - silu) + silu, and
    the oracle's d_gate equals dy * y * (either form)."""
    xs = np.linspace(-30, 30, 2001)
    s = 1 / (1 + np.exp(-xs))
    silu = xs * s
    np.testing.assert_allclose(s * (1 + xs * (1 - s)), s * (1 - silu) + silu, rtol=1e-12, atol=1e-15)
    x = _tiny_random(seed=8)
    g = oracle.bwd(x)
    out, y = oracle.fwd(x)
    sg = 1 / (1 + np.exp(-x["gate"]))
    sl = x["gate"] * sg
    np.testing.assert_allclose(g["d_gate"], x["dy"] * y * (sg * (1 - sl) + sl), rtol=1e-12, atol=1e-14)


def test_sympy_autodiff_tiny():
    """Differentiate the forward definition symbolically; compare every gradient."""
    sp = pytest.importorskip("sympy")
    batch, T, Di, N = 1, 3, 2, 2
    x = _tiny_random(seed=12, batch=batch, T=T, Di=Di, N=N)
    sym = {k: np.empty(v.shape, dtype=object) for k, v in x.items() if k != "dy"}
    subs = {}
    for k, arr in sym.items():
        for idx in np.ndindex(arr.shape):
            s = sp.Symbol(f"{k}_{'_'.join(map(str, idx))}")
            arr[idx] = s
            subs[s] = sp.Float(float(x[k][idx]), 30)
    L = 0
    for b in range(batch):
        for d in range(Di):
            h = [0] * N
            for t in range(T):
                for n in range(N):
                    a = sp.exp(sym["delta"][b, t, d] * (-sp.exp(sym["A_log"][d, n])))
                    h[n] = a * h[n] + sym["delta"][b, t, d] * sym["u"][b, t, d] * sym["B"][b, t, n]
                yv = sum(sym["C"][b, t, n] * h[n] for n in range(N)) + sym["D"][d] * sym["u"][b, t, d]
                g = sym["gate"][b, t, d]
                L += float(x["dy"][b, t, d]) * yv * g / (1 + sp.exp(-g))
    gr = oracle.bwd(x)
    for gk in GRAD_KEYS:
        arr = sym[INPUT_OF[gk]]
        for idx in np.ndindex(arr.shape):
            ref = float(sp.diff(L, arr[idx]).evalf(25, subs=subs))
            assert abs(gr[gk][idx] - ref) <= 1e-12 * max(1.0, abs(ref)), (gk, idx, gr[gk][idx], ref)


def test_row_split_threads_consistent():
    x = synth.random_inputs(3, 20, 7, 5, seed=2)
    g1 = oracle.bwd(x, threads=1)
    g4 = oracle.bwd(x, threads=4)
    for k in GRAD_KEYS:
        np.testing.assert_allclose(g4[k], g1[k], rtol=1e-13, atol=1e-13)


def test_bwd_rows_into_matches_bwd():
    # Two row ranges written into caller-owned arrays give what one bwd() call gives.
    x = synth.random_inputs(2, 9, 5, 3, seed=4)
    ref = oracle.bwd(x)
    b, T, Di, N = 2, 9, 5, 3
    per_row = {k: np.full((b, T, Di), np.nan) for k in ("d_delta", "d_u", "d_gate")}
    acc = {"d_B": np.zeros((b, T, N)), "d_C": np.zeros((b, T, N)),
           "d_A_log": np.zeros((Di, N)), "d_D": np.zeros(Di)}
    oracle.bwd_rows_into(x, (0, 4), per_row, acc)
    oracle.bwd_rows_into(x, (4, b * Di), per_row, acc)
    for k in GRAD_KEYS:
        got = per_row[k] if k in per_row else acc[k]
        np.testing.assert_allclose(got, ref[k], rtol=1e-13, atol=1e-13)


MUTANTS = {
    "carry_without_decay": ("dh[n] = da * g_h;", "dh[n] = g_h;"),
    "dropped_A_term_in_d_delta": ("ddl += g_h * (A[n] * da * hp + uu * bn);", "ddl += g_h * (uu * bn);"),
    "d_C_uses_h_prev": ("d_C_acc[bt * N + n] += dyv * hc;", "d_C_acc[bt * N + n] += dyv * hp;"),
    "wrong_sign_of_A": ("-exp(A_log[d * N + n])", "exp(A_log[d * N + n])"),
    "fwd_input_term_without_delta": ("h[n] = da * h[n] + delta[i] * u[i] * Bm[bt * N + n];",
                                     "h[n] = da * h[n] + u[i] * Bm[bt * N + n];"),
    "silu_grad_sign": ("(s * (1.0 + g * (1.0 - s)))", "(s * (1.0 - g * (1.0 - s)))"),
    "d_A_log_without_A": ("+= g_h * da * dl * A[n] * hp;", "+= g_h * da * dl * hp;"),
    "B_C_transposed_in_bwd": ("const double bn = Bm[bt * N + n];", "const double bn = Cm[bt * N + n];"),
    "d_u_skip_term_missing": ("double du = dyv * Dp[d];", "double du = 0.0;"),
    "softplus_grad_sigmoid_of_minus_x": ("d_delta[i] * (1.0 / (1.0 + exp(-raw[i])))",
                                         "d_delta[i] * (1.0 / (1.0 + exp(raw[i])))"),
    "softplus_threshold_branch_swapped": ("delta[i] = raw[i] > 20.0 ? raw[i] : log1p(exp(raw[i]));",
                                          "delta[i] = raw[i] < 20.0 ? raw[i] : log1p(exp(raw[i]));"),
    "softplus_without_log1p": ("log1p(exp(raw[i]))", "exp(raw[i])"),
    "conv_carry_taps_reversed": ("carry[k + 1] + dp * w[d * K + (K - 2 - k)];",
                                 "carry[k + 1] + dp * w[d * K + (k + 1)];"),
    "conv_carry_not_added": ("dx += carry[0];", "dx += 0.0;"),
    "conv_causal_window_shifted": ("const int64_t ts = t - (K - 1) + j;\n          if (ts >= 0) acc",
                                   "const int64_t ts = t - K + j;\n          if (ts >= 0) acc"),
    "time_index_off_by_one": ("const double hp = (t > 0) ? H[(t - 1) * N + n] : 0.0;\n        const double hc",
                              "const double hp = (t > 1) ? H[(t - 2) * N + n] : 0.0;\n        const double hc"),
}


def test_real_oracle_passes_every_pin():
    failing = [name for name, pin in PINS.items() if not pin(None)]
    assert failing == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant, tmp_path):
    find, repl = MUTANTS[mutant]
    src = oracle.source()
    assert find in src, mutant
    lib = oracle.compile_variant(src.replace(find, repl), str(tmp_path))
    failing = [name for name, pin in PINS.items() if not pin(lib)]
    assert failing, f"planted mistake {mutant} passed every pin"
