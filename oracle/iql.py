"""IQL value network, expectile loss and advantage-weighted policy (oracle side).

Follows "GPU IQL + HER Porting Plan":
  * "IQL (CPU)" item 1: V(s) is a 3-layer MLP state_dim -> hidden -> hidden
    -> 1, Linear -> ReLU -> Linear -> ReLU -> Linear, squeezed to [batch].
  * "IQL (CPU)" item 2: diff = Q(s,a) - V(s); weight = tau where diff >= 0,
    1 - tau where diff < 0; loss = mean(weight * diff^2).
  * "IQL (CPU)" item 3: A = Q - V per action; pi = softmax(beta *
    clamp(A, -10, 10)) with max-subtraction; output [batch, num_actions].
  * "CUDA Kernel: iql_value_kernel.cu": Q(s, a_taken) is the target; the
    kernel backpropagates through V into a flat gradient buffer laid out as
    w_v1, b_v1, w_v2, b_v2, w_vout, b_vout.

All arithmetic in fp64.  Linear layers are y = x W^T + b with W[out, in]
row-major.  The ReLU derivative is 1[z > 0]; the expectile weight is a
constant in the derivative, so dL/dV_b = -2 w_b d_b / B.

bf16-operand mode (forward / backward with gemm_operand=precision.bf16):
the operands of the five matrix products are rounded before the product
("Phase 2: Multi-Stream Graph Parallelism", "2C. Grouped GEMM for IQL":
bf16 GEMM inputs, fp32 accumulation); see oracle/precision.py for which
values that covers.  With gemm_operand=None the products are exact.
"""
import numpy as np


def _same(a):
    return a


def unflatten(flat, state_dim: int, hidden: int):
    """Split the flat parameter buffer into (W1, b1, W2, b2, W3, b3), fp64."""
    p = np.asarray(flat, dtype=np.float64)
    s, h = state_dim, hidden
    o = 0
    w1 = p[o:o + h * s].reshape(h, s); o += h * s
    b1 = p[o:o + h]; o += h
    w2 = p[o:o + h * h].reshape(h, h); o += h * h
    b2 = p[o:o + h]; o += h
    w3 = p[o:o + h].reshape(1, h); o += h
    b3 = p[o:o + 1]; o += 1
    assert o == p.size
    return w1, b1, w2, b2, w3, b3


def flatten(w1, b1, w2, b2, w3, b3):
    return np.concatenate([w1.ravel(), b1.ravel(), w2.ravel(), b2.ravel(), w3.ravel(), b3.ravel()])


def forward(flat, states, state_dim: int, hidden: int, gemm_operand=None):
    """V forward.  Returns V[B] and the activations the backward needs.

    gemm_operand: None, or the rounding applied to each operand of the two
    matrix products (X and W1; h1 and W2) before the product.
    """
    r = _same if gemm_operand is None else gemm_operand
    w1, b1, w2, b2, w3, b3 = unflatten(flat, state_dim, hidden)
    x = np.asarray(states, dtype=np.float64)[:, :state_dim]
    z1 = r(x) @ r(w1).T + b1
    h1 = np.maximum(z1, 0.0)
    z2 = r(h1) @ r(w2).T + b2
    h2 = np.maximum(z2, 0.0)
    v = (h2 @ w3.T + b3)[:, 0]
    return v, dict(x=x, z1=z1, h1=h1, z2=z2, h2=h2)


def iql_target(flat, next_states, rewards, dones, gamma: float, state_dim: int, hidden: int):
    """IQL bootstrap target for the Q loss and V(s').

    "GPU IQL + HER Porting Plan", "IQL modifies the target computation": the
    target r + gamma max_a Q_target(s', a') becomes r + gamma V(s'), V(s')
    from the value network's forward pass on the next states
    (forward_values).  A terminal transition (done = 1) bootstraps nothing:
    target = r + gamma (1 - done) V(s').
    """
    v, _ = forward(flat, next_states, state_dim, hidden)
    r = np.asarray(rewards, dtype=np.float64)
    d = np.asarray(dones, dtype=np.float64)
    return r + float(gamma) * (1.0 - d) * v, v


def q_taken(q, actions):
    """Q(s, a_taken): the entry of each Q row at the row's action."""
    q = np.asarray(q, dtype=np.float64)
    a = np.asarray(actions, dtype=np.int64)
    return q[np.arange(q.shape[0]), a]


def expectile_loss(qt, v, tau: float):
    """loss = mean(w * d^2), d = q - v, w = tau if d >= 0 else 1 - tau; and dL/dV."""
    qt = np.asarray(qt, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    tau = float(tau)
    d = qt - v
    w = np.where(d >= 0.0, tau, 1.0 - tau)
    n = d.shape[0]
    loss = float(np.sum(w * d * d) / n) if n else 0.0
    dv = -2.0 * w * d / n if n else np.zeros(0)
    return loss, dv


def policy(q, v, beta: float):
    """pi = softmax(beta * clamp(Q - V, -10, 10)) per row, and its argmax.

    The argmax is the lowest index among the row's maxima.
    """
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    a = np.clip(q - v[:, None], -10.0, 10.0)
    z = float(beta) * a
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    pi = e / e.sum(axis=1, keepdims=True)
    return pi, np.argmax(pi, axis=1).astype(np.int32)


def backward(flat, act: dict, dv, state_dim: int, hidden: int, gemm_operand=None):
    """Gradient of the loss w.r.t. the flat parameters, given dL/dV[B].

    gemm_operand: None, or the rounding applied to each operand of the three
    matrix products (dz2 and h1 for dW2; dz2 and W2 for dh1; dz1 and X for
    dW1) before the product.  The bias gradients (batch sums of dz1, dz2,
    dV) and dW3 (the N = 1 output layer) are not matrix products and stay
    exact.
    """
    r = _same if gemm_operand is None else gemm_operand
    w1, b1, w2, b2, w3, b3 = unflatten(flat, state_dim, hidden)
    dv = np.asarray(dv, dtype=np.float64)
    x, z1, h1, z2, h2 = act["x"], act["z1"], act["h1"], act["z2"], act["h2"]
    dh2 = dv[:, None] * w3            # [B, H]
    dz2 = dh2 * (z2 > 0.0)
    dw3 = (dv[None, :] @ h2)          # [1, H]
    db3 = np.array([dv.sum()])
    dw2 = r(dz2).T @ r(h1)            # [H, H]
    db2 = dz2.sum(axis=0)
    dh1 = r(dz2) @ r(w2)              # [B, H]
    dz1 = dh1 * (z1 > 0.0)
    dw1 = r(dz1).T @ r(x)             # [H, S]
    db1 = dz1.sum(axis=0)
    return flatten(dw1, db1, dw2, db2, dw3, db3)


def backward_abs(flat, act: dict, dv, state_dim: int, hidden: int):
    """Per gradient element, the sum of |terms| of its expanded sum.

    The backward of `backward` with every factor replaced by its absolute
    value.  |grad_i| <= backward_abs_i, with equality when every term of
    element i has one sign.  Rounding error of any summation order of
    element i is bounded by a multiple of backward_abs_i, so elements with
    |grad_i| far below it have a sign that finite precision does not fix.
    """
    w1, b1, w2, b2, w3, b3 = unflatten(flat, state_dim, hidden)
    adv = np.abs(np.asarray(dv, dtype=np.float64))
    x, z1, h1, z2, h2 = act["x"], act["z1"], act["h1"], act["z2"], act["h2"]
    adz2 = adv[:, None] * np.abs(w3) * (z2 > 0.0)
    adw3 = adv[None, :] @ np.abs(h2)
    adb3 = np.array([adv.sum()])
    adw2 = adz2.T @ np.abs(h1)
    adb2 = adz2.sum(axis=0)
    adz1 = (adz2 @ np.abs(w2)) * (z1 > 0.0)
    adw1 = adz1.T @ np.abs(x)
    adb1 = adz1.sum(axis=0)
    return flatten(adw1, adb1, adw2, adb2, adw3, adb3)


def value_fwd_bwd(flat, states, qt, tau: float, state_dim: int, hidden: int, gemm_operand=None):
    """V forward + expectile loss + backward, as one call (fp64 sums)."""
    v, act = forward(flat, states, state_dim, hidden, gemm_operand)
    loss, dv = expectile_loss(qt, v, tau)
    grad = backward(flat, act, dv, state_dim, hidden, gemm_operand)
    return v, loss, grad
