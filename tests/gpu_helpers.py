"""Helpers shared by the GPU parity tests (tolerances and transfers)."""
import numpy as np

import oracle
import synthetic as syn


def dev_tensor(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def gemv_tol(fmt, W, r0, r1, in_dim, x):
    """Per-row bound max|y_gpu - y_ref| <= 1e-3 * ||W_r||_2 * ||x||_2."""
    return 1e-3 * oracle.row_norms(fmt, W, r0, r1, in_dim) * float(
        np.linalg.norm(np.asarray(x, dtype=np.float64)))


def assert_gemv_close(y_gpu, y_ref, tol, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, (f"{what}: {bad.size} rows out of tolerance, first row {bad[0]}: "
                           f"gpu {y_gpu[bad[0]]} ref {y_ref[bad[0]]} tol {tol[bad[0]]}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0


def swiglu_h_tol(g_ref, u_ref, tg, tu):
    """Bound on |h_gpu - h_ref| for h = silu(g)*u given |dg| <= tg, |du| <= tu:
    |silu'| <= 1.1, plus fp32 rounding of the epilogue."""
    silu = g_ref / (1.0 + np.exp(-g_ref))
    return 1.1 * tg * (np.abs(u_ref) + tu) + np.abs(silu) * tu + 1e-6 * np.abs(silu * u_ref)


def moe_reference(fmt, G, U, D, n_ff, n_embd, x, logits, top_k):
    """The routed SwiGLU FFN computed by the oracle alone (nothing from the
    CUDA path goes in), with bounds derived from the per-GEMV tolerance:
      h_k = silu(G_k x) * (U_k x)     within swiglu_h_tol of the GPU's h_k;
      y   = sum_k w_k D_k h_k         the GPU's down GEMV runs on its own h_k,
            so per row |dy| <= sum_k w_k (1e-3 ||D_k,r|| (||h_k|| + ||dh_k||)
                                          + ||D_k,r|| ||dh_k||)
            (Cauchy-Schwarz on the h error), plus fp32 rounding of the
            router weights and the weighted sum (1e-6 relative).
    Returns a dict with idx, w, h (list), tol_h (list), y, tol_y."""
    idx, w = oracle.router_topk(logits, top_k)
    y = np.zeros(n_embd)
    tol_y = np.zeros(n_embd)
    hs, ths = [], []
    for k, e in enumerate(idx):
        e = int(e)
        Ge, Ue = G[e * n_ff:(e + 1) * n_ff], U[e * n_ff:(e + 1) * n_ff]
        De = D[e * n_embd:(e + 1) * n_embd]
        g = oracle.gemv(fmt, Ge, 0, n_ff, n_embd, x)
        u = oracle.gemv(fmt, Ue, 0, n_ff, n_embd, x)
        h = oracle.silu_vec(g) * u
        th = swiglu_h_tol(g, u, gemv_tol(fmt, Ge, 0, n_ff, n_embd, x),
                          gemv_tol(fmt, Ue, 0, n_ff, n_embd, x))
        yk = oracle.gemv(fmt, De, 0, n_embd, n_ff, h)
        nD = oracle.row_norms(fmt, De, 0, n_embd, n_ff)
        nh, nth = float(np.linalg.norm(h)), float(np.linalg.norm(th))
        y += float(w[k]) * yk
        tol_y += float(w[k]) * (1e-3 * nD * (nh + nth) + nD * nth) + 1e-6 * np.abs(yk)
        hs.append(h)
        ths.append(th)
    return {"idx": idx, "w": w, "h": hs, "tol_h": ths, "y": y, "tol_y": tol_y}


def check_moe(ref, y, idx=None, w=None, h=None, what=""):
    """Compares a GPU MoE result (and, when given, its routing and h) with
    moe_reference: indices equal, weights within fp32 rounding, h and y
    within the derived bounds."""
    if idx is not None:
        assert list(np.asarray(idx).tolist()) == list(ref["idx"].tolist()), f"{what}: routing"
    if w is not None:
        np.testing.assert_allclose(np.asarray(w, np.float64), ref["w"], rtol=1e-5, atol=1e-7)
    if h is not None:
        for k in range(len(ref["h"])):
            assert_gemv_close(np.asarray(h[k]), ref["h"][k], ref["tol_h"][k], f"{what}: h[{k}]")
    assert_gemv_close(np.asarray(y), ref["y"], ref["tol_y"], f"{what}: y")


# |d/dz gelu(z)| = |Phi(z) + z phi(z)| <= 1.129 (its maximum, at z = sqrt(2))
GELU_SLOPE_MAX = 1.13


def chained_y_tol(fmt, Dm, rows, in_dim, h, th):
    """Bound on |y_gpu - D h_ref| per row of D (rows: a list) when the GPU's
    down GEMV runs on its own h = h_ref + dh with |dh| <= th elementwise:
    1e-3 ||D_r|| ||h_gpu|| + ||D_r|| ||dh|| <= ||D_r|| (1e-3 (||h|| + ||th||)
    + ||th||) (Cauchy-Schwarz)."""
    nD = np.array([oracle.row_norms(fmt, Dm, int(r), int(r) + 1, in_dim)[0] for r in rows])
    nh, nth = float(np.linalg.norm(h)), float(np.linalg.norm(th))
    return nD * (1e-3 * (nh + nth) + nth)


def ffn_reference(fmt, G, U, D, n_ff, n_embd, x, act="swiglu", rows=None):
    """The two-phase FFN by the oracle alone (no GPU value goes in):
    swiglu: h = silu(G x) * (U x); gelu: h = gelu(U x) (G unused); then
    y[r] = D_r . h for r in rows (default all).  Returns h, its bound tol_h,
    y and its bound tol_y, derived from the per-GEMV tolerance."""
    u = oracle.gemv(fmt, U, 0, n_ff, n_embd, x)
    tu = gemv_tol(fmt, U, 0, n_ff, n_embd, x)
    if act == "swiglu":
        g = oracle.gemv(fmt, G, 0, n_ff, n_embd, x)
        h = oracle.silu_vec(g) * u
        th = swiglu_h_tol(g, u, gemv_tol(fmt, G, 0, n_ff, n_embd, x), tu)
    else:
        h = oracle.gelu_vec(u)
        th = GELU_SLOPE_MAX * tu + 1e-6 * np.abs(h)
    rows = list(range(n_embd)) if rows is None else [int(r) for r in rows]
    y = np.array([oracle.gemv(fmt, D, r, r + 1, n_ff, h)[0] for r in rows]) if len(rows) < n_embd \
        else oracle.gemv(fmt, D, 0, n_embd, n_ff, h)
    tol_y = chained_y_tol(fmt, D, rows, n_ff, h, th) + 1e-6 * np.abs(y)
    return {"u": u, "tol_u": tu, "h": h, "tol_h": th, "y": y, "tol_y": tol_y, "rows": rows}


def swiglu_clamped_h_tol(g, u, tg, tu, alpha, limit):
    """Bound on |h_gpu - h_ref| for the clamped SwiGLU h = f(g') (u' + 1),
    f(z) = z sigmoid(alpha z), g' = min(g, limit), u' = clamp(u, +-limit),
    given |dg| <= tg, |du| <= tu: both clamps are 1-Lipschitz and
    |f'| <= 1.1 for every alpha (f'(z) = s(t) + t s(t)(1 - s(t)), t = alpha z,
    whose maximum is 1.0998), so |dh| <= 1.1 tg (|u' + 1| + tu) + |f(g')| tu,
    plus fp32 rounding of the epilogue."""
    gc, uc = np.minimum(g, limit), np.clip(u, -limit, limit)
    f = gc / (1.0 + np.exp(-alpha * gc))
    return 1.1 * tg * (np.abs(uc + 1.0) + tu) + np.abs(f) * tu + 1e-6 * np.abs(f * (uc + 1.0))


def moe_reference_biased(fmt, G, U, D, n_ff, n_embd, x, logits, top_k, gate_bias, up_bias,
                         down_bias, alpha, limit):
    """moe_reference for the biased experts with the clamped SwiGLU: y and h
    from the oracle's own chain (oracle.moe_ffn_biased), bounds derived from
    the per-GEMV tolerance (the fp32 bias additions add 1e-7 relative)."""
    y, idx, w, h = oracle.moe_ffn_biased(fmt, logits, top_k, G, U, D, gate_bias, up_bias,
                                         down_bias, alpha, limit, n_ff, n_embd, x)
    tol_y = np.zeros(n_embd)
    hs, ths = [], []
    clamped = 0   # gate or up values the clamp changed
    for k, e in enumerate(idx):
        e = int(e)
        Ge, Ue = G[e * n_ff:(e + 1) * n_ff], U[e * n_ff:(e + 1) * n_ff]
        De = D[e * n_embd:(e + 1) * n_embd]
        bg = 0.0 if gate_bias is None else np.asarray(gate_bias, np.float64)[e]
        bu = 0.0 if up_bias is None else np.asarray(up_bias, np.float64)[e]
        g = oracle.gemv(fmt, Ge, 0, n_ff, n_embd, x) + bg
        u = oracle.gemv(fmt, Ue, 0, n_ff, n_embd, x) + bu
        tg = gemv_tol(fmt, Ge, 0, n_ff, n_embd, x) + 1e-7 * np.abs(g)
        tu = gemv_tol(fmt, Ue, 0, n_ff, n_embd, x) + 1e-7 * np.abs(u)
        th = swiglu_clamped_h_tol(g, u, tg, tu, alpha, limit)
        clamped += int((g > limit).sum() + (np.abs(u) > limit).sum())
        yk = oracle.gemv(fmt, De, 0, n_embd, n_ff, h[k])
        bd = 0.0 if down_bias is None else np.asarray(down_bias, np.float64)[e]
        tol_y += float(w[k]) * (chained_y_tol(fmt, De, range(n_embd), n_ff, h[k], th)
                                + 1e-6 * (np.abs(yk) + np.abs(bd)))
        hs.append(h[k])
        ths.append(th)
    return {"idx": idx, "w": w, "h": hs, "tol_h": ths, "y": y, "tol_y": tol_y,
            "clamped": clamped}


def derived_gemm_bound(fmt, W, r0, r1, in_dim, X):
    """(n_tok, rows) error bound of rf_gemm's arithmetic, from the oracle's
    exact dequantized weights: w and x each rounded once to fp16 (relative
    2^-11, absolute 2^-25 below the normal range), fp16 x fp16 products exact
    in fp32, fp32 accumulation over in_dim terms bounded loosely by
    in_dim * 2^-23 times the sum of |products| (truncating adds allowed);
    Q4_K's weights take one fp32 rounding first (another 2^-23)."""
    Wd = oracle.dequantize(fmt, W[r0:r1]).astype(np.float64).reshape(r1 - r0, in_dim)
    Xa = np.abs(np.asarray(X, dtype=np.float64))
    Wa = np.abs(Wd)
    S = Xa @ Wa.T
    lin = 2.0 ** -25 * 1.001 * (Wa.sum(axis=1)[None, :] + Xa.sum(axis=1)[:, None])
    extra = 2.0 ** -23 if fmt == syn.Q4_K else 0.0
    return (2.0 ** -10 + 2.0 ** -22 + extra + in_dim * 2.0 ** -23) * S + lin
