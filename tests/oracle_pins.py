"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an oracle library handle and returns a list of
failure strings (empty = pass).  The tests call them against the real oracle,
and against copies of it with a planted mistake, to show every pin battery
catches those mistakes.

Sources of the facts:
  * the definition in the forward kernel of "flash_attention_2.cu"
    (leloykun/flash-hyperbolic-attention-minimal), evaluated independently at
    50 digits with Python's ``decimal`` (no max shift, no tiling);
  * closed forms that follow from it (constant V, one key, causal row 0,
    uniform scores, hand-derived worked examples under tests/golden/);
  * invariants (linearity in V, joint K/V permutation, score shift);
  * a library special case: torch's float64 scaled_dot_product_attention.
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "closed_form_cases.json")


def _close(a, b, rtol, atol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.shape != b.shape:
        return False
    return bool(np.all(np.abs(a - b) <= atol + rtol * np.abs(b)))


# ---------------------------------------------------------------- decimal
def decimal_attention(q, k, v, scale, causal, prec=50):
    """The definition evaluated with Decimal: w_j = exp(s_j), no max shift."""
    getcontext().prec = prec
    B, H, Nq, d = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    o = np.zeros((B, H, Nq, dv))
    lse = np.zeros((B, H, Nq))
    sc = Decimal(repr(float(scale)))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                keys = range(min(i + 1, Nk)) if causal else range(Nk)
                ws, num = [], [Decimal(0)] * dv
                for j in keys:
                    dot = sum(Decimal(repr(float(q[b, h, i, x]))) *
                              Decimal(repr(float(k[b, h, j, x]))) for x in range(d))
                    w = (sc * dot).exp()
                    ws.append(w)
                    for x in range(dv):
                        num[x] += w * Decimal(repr(float(v[b, h, j, x])))
                tot = sum(ws)
                for x in range(dv):
                    o[b, h, i, x] = float(num[x] / tot)
                lse[b, h, i] = float(tot.ln())
    return o, lse


def _rand_int(rng, shape, lo=-2, hi=2):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


# ---------------------------------------------------------------- pins
def pin_golden(lib):
    """Hand-derived worked examples (tests/golden/closed_form_cases.json)."""
    fails = []
    getcontext().prec = 50
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    e = Decimal(1).exp()
    env = {"e": e, "exp": lambda x: Decimal(x).exp(), "ln": lambda x: Decimal(x).ln(),
           "__builtins__": {}}
    for c in cases:
        q = np.array(c["q"], np.float32)[None, None]
        k = np.array(c["k"], np.float32)[None, None]
        v = np.array(c["v"], np.float32)[None, None]
        o, lse = oracle.attn_fwd(q, k, v, c["scale"], c["causal"], lib=lib)
        eo = np.array([[float(eval(s, env)) for s in row] for row in c["expect_o"]])
        el = np.array([float(eval(s, env)) for s in c["expect_lse"]])
        if not _close(o[0, 0], eo, 1e-14, 1e-14):
            fails.append(f"golden {c['name']}: O {o[0, 0].tolist()} != {eo.tolist()}")
        if not _close(lse[0, 0], el, 1e-14, 1e-14):
            fails.append(f"golden {c['name']}: LSE {lse[0, 0].tolist()} != {el.tolist()}")
    return fails


def pin_brute_force(lib, seed=1):
    """Tiny integer inputs against the 50-digit definition."""
    fails = []
    rng = np.random.default_rng(seed)
    shapes = [(1, 1, 1, 1, 1), (1, 1, 2, 2, 2), (1, 2, 3, 3, 4), (2, 1, 5, 5, 2),
              (1, 1, 5, 3, 4), (1, 1, 2, 5, 1), (1, 2, 4, 7, 3)]
    for (B, H, Nq, Nk, d) in shapes:
        for scale in (1.0, 0.5, -0.75):
            for causal in (False, True):
                q = _rand_int(rng, (B, H, Nq, d))
                k = _rand_int(rng, (B, H, Nk, d))
                v = _rand_int(rng, (B, H, Nk, d), -3, 3)
                o, lse = oracle.attn_fwd(q, k, v, scale, causal, lib=lib)
                eo, el = decimal_attention(q, k, v, scale, causal)
                tag = f"brute {B,H,Nq,Nk,d} scale={scale} causal={causal}"
                if not _close(o, eo, 1e-13, 1e-13):
                    fails.append(f"{tag}: O max err {np.max(np.abs(o - eo)):.3e}")
                if not _close(lse, el, 1e-13, 1e-13):
                    fails.append(f"{tag}: LSE max err {np.max(np.abs(lse - el)):.3e}")
    return fails


def pin_probs(lib, seed=2):
    """Every probability row sums to 1; masked keys get exactly 0; the
    probabilities themselves match the 50-digit definition."""
    fails = []
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        for (Nq, Nk) in ((4, 4), (6, 3), (3, 6)):
            q = rng.standard_normal((1, 2, Nq, 3)).astype(np.float32)
            k = rng.standard_normal((1, 2, Nk, 3)).astype(np.float32)
            p = oracle.attn_probs(q, k, 0.7, causal, lib=lib)
            if not np.all(np.abs(p.sum(-1) - 1.0) <= 1e-14):
                fails.append(f"probs causal={causal} {Nq}x{Nk}: rows do not sum to 1")
            if causal:
                i = np.arange(Nq)[:, None]
                j = np.arange(Nk)[None, :]
                if np.any(p[..., (j > i)] != 0.0):
                    fails.append(f"probs causal {Nq}x{Nk}: a key j > i has weight")
            # P V with V = identity columns reproduces P: compare to decimal
            eye = np.zeros((1, 2, Nk, Nk), np.float32)
            eye[..., np.arange(Nk), np.arange(Nk)] = 1.0
            eo, _ = decimal_attention(q, k, eye, 0.7, causal)
            if not _close(p, eo, 1e-13, 1e-14):
                fails.append(f"probs causal={causal} {Nq}x{Nk}: P != decimal softmax")
    return fails


def pin_constant_v(lib, seed=3):
    """If every value row is the same vector c, every output row is c."""
    fails = []
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        q = rng.standard_normal((2, 2, 9, 5)).astype(np.float32)
        k = rng.standard_normal((2, 2, 7, 5)).astype(np.float32)
        c = rng.standard_normal(5).astype(np.float32)
        v = np.broadcast_to(c, (2, 2, 7, 5)).copy()
        o, _ = oracle.attn_fwd(q, k, v, 0.9, causal, lib=lib)
        if not _close(o, np.broadcast_to(c.astype(np.float64), o.shape), 1e-13, 1e-13):
            fails.append(f"constant V causal={causal}: O != c")
    return fails


def pin_causal_row0(lib, seed=4):
    """Causal: query 0 sees key 0 only, so O[0] = V[0] and LSE[0] = scale*q0.k0."""
    fails = []
    rng = np.random.default_rng(seed)
    q = _rand_int(rng, (2, 3, 6, 4))
    k = _rand_int(rng, (2, 3, 6, 4))
    v = rng.standard_normal((2, 3, 6, 4)).astype(np.float32)
    o, lse = oracle.attn_fwd(q, k, v, 0.25, True, lib=lib)
    if not _close(o[:, :, 0], v[:, :, 0].astype(np.float64), 0, 1e-15):
        fails.append("causal row 0: O[0] != V[0]")
    want = 0.25 * np.einsum("bhx,bhx->bh", q[:, :, 0].astype(np.float64),
                            k[:, :, 0].astype(np.float64))
    if not _close(lse[:, :, 0], want, 0, 1e-13):
        fails.append("causal row 0: LSE[0] != scale*q0.k0")
    return fails


def pin_single_key(lib, seed=5):
    """Nk = 1: every row returns V[0] and LSE[i] = scale*q_i.k_0."""
    fails = []
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        q = _rand_int(rng, (1, 2, 5, 3))
        k = _rand_int(rng, (1, 2, 1, 3))
        v = rng.standard_normal((1, 2, 1, 3)).astype(np.float32)
        o, lse = oracle.attn_fwd(q, k, v, 1.5, causal, lib=lib)
        if not _close(o, np.broadcast_to(v.astype(np.float64), o.shape), 0, 1e-15):
            fails.append(f"one key causal={causal}: O != V[0]")
        want = 1.5 * np.einsum("bhix,bhx->bhi", q.astype(np.float64),
                               k[:, :, 0].astype(np.float64))
        if not _close(lse, want, 0, 1e-13):
            fails.append(f"one key causal={causal}: LSE != scale*q.k0")
    return fails


def pin_uniform(lib, seed=6):
    """scale = 0: all allowed keys weigh the same, so O[i] is the mean of the
    allowed value rows (a prefix mean when causal) and LSE[i] = ln |K(i)|."""
    fails = []
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        Nq, Nk = 7, 5
        q = rng.standard_normal((1, 2, Nq, 3)).astype(np.float32)
        k = rng.standard_normal((1, 2, Nk, 3)).astype(np.float32)
        v = rng.standard_normal((1, 2, Nk, 3)).astype(np.float32)
        o, lse = oracle.attn_fwd(q, k, v, 0.0, causal, lib=lib)
        for i in range(Nq):
            n = min(i + 1, Nk) if causal else Nk
            want = v[:, :, :n].astype(np.float64).mean(axis=2)
            if not _close(o[:, :, i], want, 1e-13, 1e-14):
                fails.append(f"uniform causal={causal}: O[{i}] != mean of {n} rows")
            if not _close(lse[:, :, i], np.full((1, 2), math.log(n)), 1e-14, 1e-15):
                fails.append(f"uniform causal={causal}: LSE[{i}] != ln {n}")
    return fails


def pin_invariants(lib, seed=7):
    """Linearity in V; joint permutation of keys and values (non-causal);
    permutation of queries (non-causal); shifting every key by the same
    vector c moves every score of row i by scale*q_i.c, leaving O unchanged
    and adding scale*q_i.c to LSE."""
    fails = []
    rng = np.random.default_rng(seed)
    q = _rand_int(rng, (2, 2, 6, 4))
    k = _rand_int(rng, (2, 2, 8, 4))
    v1 = rng.standard_normal((2, 2, 8, 4)).astype(np.float32)
    v2 = rng.standard_normal((2, 2, 8, 4)).astype(np.float32)
    for causal in (False, True):
        o1, _ = oracle.attn_fwd(q, k, v1, 0.6, causal, lib=lib)
        o2, _ = oracle.attn_fwd(q, k, v2, 0.6, causal, lib=lib)
        # 2*v1 + v2 is exact in float32 for these magnitudes? not always: use
        # powers of two so the combination is exact.
        v3 = (np.float32(2.0) * v1 + v2).astype(np.float32)
        o3, _ = oracle.attn_fwd(q, k, v3, 0.6, causal, lib=lib)
        lin = 2.0 * o1 + o2
        v3err = (v3.astype(np.float64) - (2.0 * v1.astype(np.float64) + v2)).max()
        if not _close(o3, lin, 1e-12, 1e-12 + 4 * abs(v3err)):
            fails.append(f"linearity causal={causal}")
    perm = rng.permutation(8)
    o, lse = oracle.attn_fwd(q, k, v1, 0.6, False, lib=lib)
    op, lsep = oracle.attn_fwd(q, k[:, :, perm], v1[:, :, perm], 0.6, False, lib=lib)
    if not (_close(op, o, 1e-13, 1e-13) and _close(lsep, lse, 1e-13, 1e-13)):
        fails.append("joint K/V permutation changed the result")
    qperm = rng.permutation(6)
    oq, lseq = oracle.attn_fwd(q[:, :, qperm], k, v1, 0.6, False, lib=lib)
    if not (_close(oq, o[:, :, qperm], 0, 0) and _close(lseq, lse[:, :, qperm], 0, 0)):
        fails.append("query permutation did not permute the rows")
    for causal in (False, True):
        c = np.array([1, -2, 0, 3], np.float32)
        o, lse = oracle.attn_fwd(q, k, v1, 0.5, causal, lib=lib)
        os_, lses = oracle.attn_fwd(q, k + c, v1, 0.5, causal, lib=lib)
        shift = 0.5 * np.einsum("bhix,x->bhi", q.astype(np.float64), c.astype(np.float64))
        if not _close(os_, o, 1e-12, 1e-12):
            fails.append(f"key shift changed O causal={causal}")
        if not _close(lses, lse + shift, 1e-13, 1e-12):
            fails.append(f"key shift: LSE not moved by scale*q.c causal={causal}")
    return fails


def pin_online_recurrence(lib, seed=8):
    """The tiled online-softmax recurrence (m, l, O rescaled per tile) equals
    the two-pass definition, for several tile widths and ragged lengths."""
    fails = []
    rng = np.random.default_rng(seed)
    for (Nq, Nk) in ((130, 130), (77, 301), (300, 45)):
        q = rng.standard_normal((1, 2, Nq, 16)).astype(np.float32) * 2
        k = rng.standard_normal((1, 2, Nk, 16)).astype(np.float32) * 2
        v = rng.standard_normal((1, 2, Nk, 16)).astype(np.float32)
        for causal in (False, True):
            o, lse = oracle.attn_fwd(q, k, v, 0.35, causal, lib=lib)
            for bc in (1, 7, 64, 128):
                ot, lset = oracle.attn_fwd_online(q, k, v, 0.35, causal, bc, lib=lib)
                if not (_close(ot, o, 1e-12, 1e-12) and _close(lset, lse, 1e-12, 1e-12)):
                    fails.append(f"online bc={bc} {Nq}x{Nk} causal={causal} differs")
    return fails


def pin_torch_sdpa(lib, seed=9):
    """torch's float64 CPU scaled_dot_product_attention (top-left is_causal)
    and torch.logsumexp of the masked scaled scores agree with the oracle."""
    import torch
    fails = []
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((2, 3, 64, 16)).astype(np.float32)
    k = rng.standard_normal((2, 3, 64, 16)).astype(np.float32)
    v = rng.standard_normal((2, 3, 64, 16)).astype(np.float32)
    tq, tk, tv = (torch.from_numpy(a).double() for a in (q, k, v))
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, 0.25, causal, lib=lib)
        to = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=0.25).numpy()
        s = 0.25 * (tq @ tk.transpose(-1, -2))
        if causal:
            s = s.masked_fill(torch.ones(64, 64, dtype=torch.bool).triu(1), float("-inf"))
        tl = torch.logsumexp(s, dim=-1).numpy()
        if not _close(o, to, 1e-12, 1e-12):
            fails.append(f"sdpa O causal={causal}: {np.max(np.abs(o - to)):.2e}")
        if not _close(lse, tl, 1e-12, 1e-12):
            fails.append(f"logsumexp causal={causal}: {np.max(np.abs(lse - tl)):.2e}")
    return fails


def pin_rows_api(lib, seed=10):
    """The row-sampling entry point returns exactly the full result's rows."""
    fails = []
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((2, 2, 33, 8)).astype(np.float32)
    k = rng.standard_normal((2, 2, 40, 8)).astype(np.float32)
    v = rng.standard_normal((2, 2, 40, 8)).astype(np.float32)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, 0.3, causal, lib=lib)
        rows = rng.choice(2 * 2 * 33, size=25, replace=False)
        ro, rl = oracle.attn_rows(q, k, v, rows, 0.3, causal, lib=lib)
        if not (_close(ro, o.reshape(-1, 8)[rows], 0, 0)
                and _close(rl, lse.reshape(-1)[rows], 0, 0)):
            fails.append(f"rows API causal={causal} differs from the full result")
    return fails


def pin_bwd_finite_differences(lib, seed=11):
    """dL/dq, dL/dk, dL/dv of L = sum(O * G) by central differences of the
    forward oracle, Richardson-extrapolated from steps 2^-6 and 2^-7.  Inputs
    are multiples of 1/8, so every perturbed value is exact in float32."""
    fails = []
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        q = (rng.integers(-12, 13, (1, 2, 4, 3)) / 8).astype(np.float32)
        k = (rng.integers(-12, 13, (1, 2, 5, 3)) / 8).astype(np.float32)
        v = (rng.integers(-12, 13, (1, 2, 5, 3)) / 8).astype(np.float32)
        g = rng.standard_normal((1, 2, 4, 3))
        dq, dk, dv = oracle.attn_bwd(q, k, v, g.astype(np.float32), 0.75, causal, lib=lib)
        # the oracle's dO must be the float32 G the loss uses
        g = g.astype(np.float32).astype(np.float64)

        def loss(qq, kk, vv):
            o, _ = oracle.attn_fwd(qq, kk, vv, 0.75, causal, lib=lib)
            return float(np.sum(o * g))

        for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in np.ndindex(arr.shape):
                est = []
                for h in (2.0 ** -6, 2.0 ** -7):
                    plus, minus = arr.copy(), arr.copy()
                    plus[idx] += np.float32(h)
                    minus[idx] -= np.float32(h)
                    args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
                    if name == "q":
                        lp, lm = loss(plus, k, v), loss(minus, k, v)
                    elif name == "k":
                        lp, lm = loss(q, plus, v), loss(q, minus, v)
                    else:
                        lp, lm = loss(q, k, plus), loss(q, k, minus)
                    est.append((lp - lm) / (2 * h))
                fd = (4 * est[1] - est[0]) / 3
                if abs(fd - grad[idx]) > 1e-7 + 1e-6 * abs(grad[idx]):
                    fails.append(f"bwd FD causal={causal} d{name}{idx}: {grad[idx]} vs {fd}")
    return fails


def pin_bwd_torch(lib, seed=12):
    """torch float64 autograd through scaled_dot_product_attention."""
    import torch
    fails = []
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.standard_normal((2, 2, 40, 8)).astype(np.float32) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.3, causal, lib=lib)
        tq, tk, tv = (torch.from_numpy(a).double().requires_grad_() for a in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                               scale=0.3)
        out.backward(torch.from_numpy(g).double())
        for name, a, t in (("dq", dq, tq), ("dk", dk, tk), ("dv", dv, tv)):
            if not _close(a, t.grad.numpy(), 1e-11, 1e-11):
                fails.append(f"bwd torch causal={causal} {name}: "
                             f"{np.max(np.abs(a - t.grad.numpy())):.2e}")
    return fails


def pin_bwd_identities(lib, seed=13):
    """Every row of dS sums to zero (the probabilities sum to one), so the key
    gradients sum to zero over keys and a constant key row gives dQ = 0; and
    the value gradients sum to the summed upstream gradient."""
    fails = []
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.standard_normal((1, 3, 9, 4)).astype(np.float32) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.6, causal, lib=lib)
        if not np.all(np.abs(dk.sum(axis=2)) <= 1e-13):
            fails.append(f"bwd identity causal={causal}: sum_j dK_j != 0")
        if not _close(dv.sum(axis=2), g.astype(np.float64).sum(axis=2), 1e-13, 1e-13):
            fails.append(f"bwd identity causal={causal}: sum_j dV_j != sum_i dO_i")
        kc = np.broadcast_to(k[:, :, :1], k.shape).copy()
        dq0, _, _ = oracle.attn_bwd(q, kc, v, g, 0.6, causal, lib=lib)
        if not np.all(np.abs(dq0) <= 1e-13):
            fails.append(f"bwd identity causal={causal}: constant keys but dQ != 0")
    return fails


ALL_PINS = [pin_golden, pin_brute_force, pin_probs, pin_constant_v, pin_causal_row0,
            pin_single_key, pin_uniform, pin_invariants, pin_online_recurrence,
            pin_torch_sdpa, pin_rows_api, pin_bwd_finite_differences, pin_bwd_torch,
            pin_bwd_identities]
