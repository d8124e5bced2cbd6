"""Budgeted per-source clipping and the Adam update (oracle side).

Follows:
  * "Gradient Stability -- Multi-Task Gradient Isolation + Full Spectral
    Norm", "Proper design": each gradient source gets a budget fraction of
    max_grad_norm (0.70 primary, 0.15, 0.10, 0.05; they sum to 1.0).  The
    pipeline sets grad = primary, clips it in place to its budget, then adds
    alpha * clip(source_k, budget_k) for every auxiliary source, and ends with
    Adam whose own clip at max_grad_norm should never fire.  The clipped
    SAXPY (Task 1, Step 5) computes the source norm first, then adds.
  * "DQN Backward-Path NaN Audit", the Adam kernel findings: the norm is kept
    as a raw sum of squares and square-rooted at the point of use; the clip
    scale is (n > c && n > 0) ? c / n : 1; a non-finite gradient element is
    skipped; bias correction divides by 1 - beta^t with t >= 1.
  * "GPU IQL + HER Porting Plan", "CUDA Kernel: iql_adam_kernel.cu (REUSE)":
    the Adam launch takes params, grads, m, v, t, n, lr, beta1, beta2, eps,
    weight_decay, max_grad_norm.

  * "DQN Backward-Path NaN Audit", proposed guards: an isfinite guard on
    the SAXPY (a non-finite source element adds nothing) and a bound on
    |weight| applied by the Adam kernel after its update (0 disables it).

Readings (listed in the design notes): weight decay is decoupled,
p -= lr * (m_hat / (sqrt(v_hat) + eps) + weight_decay * p); beta1, beta2 and
eps default to 0.9, 0.999, 1e-8; the clip scale follows the formula with IEEE
semantics, so a NaN norm gives scale 1 and an infinite norm gives scale 0.
"""
import numpy as np

BUDGET = (0.70, 0.15, 0.10, 0.05)


def l2norm(x) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.sum(x * x)))


def clip_scale(n: float, c: float) -> float:
    """(n > c && n > 0) ? c / n : 1 (a NaN n compares false and gives 1)."""
    return c / n if (n > c and n > 0.0) else 1.0


def sanitize(x):
    """Non-finite elements replaced by 0 (the SAXPY's isfinite guard)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(np.isfinite(x), x, 0.0)


def budgeted_combine(sources, budget_frac, alpha, max_grad_norm: float, sanitize_sources: bool = False):
    """G = sum_k alpha_k * clip(g_k, budget_frac_k * max_grad_norm).

    sources[0] is the primary gradient.  Returns (G, norms) with norms =
    [||g_0||, ..., ||g_{n-1}||, ||G||].  With sanitize_sources, every
    source's non-finite elements count as 0 in its norm and in the sum.
    """
    srcs = [np.asarray(s, dtype=np.float64) for s in sources]
    if sanitize_sources:
        srcs = [sanitize(s) for s in srcs]
    norms = [l2norm(s) for s in srcs]
    g = np.zeros_like(srcs[0])
    with np.errstate(invalid="ignore", over="ignore"):
        for k, s in enumerate(srcs):
            c = float(budget_frac[k]) * float(max_grad_norm)
            g = g + float(alpha[k]) * clip_scale(norms[k], c) * s
    norms.append(l2norm(g))
    return g, np.array(norms)


def adam(p, g, m, v, t: int, lr: float, beta1: float, beta2: float, eps: float,
         weight_decay: float, max_grad_norm: float, grad_norm: float, weight_clamp: float = 0.0):
    """One Adam step on flat buffers, with the safety clip at max_grad_norm.

    `grad_norm` is ||g|| (the combined norm).  Elements whose clipped gradient
    is not finite are left unchanged (p, m, v) and counted.  With
    weight_clamp > 0 every updated weight is then clamped to
    [-weight_clamp, weight_clamp].  Returns (p, m, v, skipped).
    """
    assert t >= 1
    p = np.asarray(p, dtype=np.float64).copy()
    m = np.asarray(m, dtype=np.float64).copy()
    v = np.asarray(v, dtype=np.float64).copy()
    s = clip_scale(float(grad_norm), float(max_grad_norm))
    with np.errstate(invalid="ignore", over="ignore"):
        gs = np.asarray(g, dtype=np.float64) * s
    ok = np.isfinite(gs)
    gk = gs[ok]
    b1, b2 = float(beta1), float(beta2)
    m[ok] = b1 * m[ok] + (1.0 - b1) * gk
    v[ok] = b2 * v[ok] + (1.0 - b2) * gk * gk
    mhat = m[ok] / (1.0 - b1 ** t)
    vhat = v[ok] / (1.0 - b2 ** t)
    p[ok] = p[ok] - float(lr) * (mhat / (np.sqrt(vhat) + float(eps)) + float(weight_decay) * p[ok])
    if weight_clamp > 0.0:
        p[ok] = np.clip(p[ok], -float(weight_clamp), float(weight_clamp))
    return p, m, v, int((~ok).sum())


def polyak(target, params, rate: float):
    """Polyak (EMA) update of a target network: (1 - rate) target + rate params
    ("GPU IQL + HER Porting Plan", target_ema_update)."""
    t = np.asarray(target, dtype=np.float64)
    return (1.0 - float(rate)) * t + float(rate) * np.asarray(params, dtype=np.float64)
