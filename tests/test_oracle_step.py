"""Pin for the oracle's composed train step against an independent torch build.

The torch side derives the gradient by autograd, clips with
torch.nn.utils.clip_grad_norm_ (whose scale has a +1e-6 in the denominator,
hence the tolerance) and updates with torch.optim.AdamW.
"""
import dataclasses

import numpy as np
import torch

import synth
from oracle import her, step


def _torch_step(w, params_t, opt, batch, q, tau, aux):
    s, h = w.state_dim, w.hidden
    t = params_t
    o = 0
    w1 = t[o:o + h * s].view(h, s); o += h * s
    b1 = t[o:o + h]; o += h
    w2 = t[o:o + h * h].view(h, h); o += h * h
    b2 = t[o:o + h]; o += h
    w3 = t[o:o + h].view(1, h); o += h
    b3 = t[o:o + 1]
    x = torch.tensor(batch["states"][:, :s], dtype=torch.float64)
    lin = torch.nn.functional.linear
    v = lin(torch.relu(lin(torch.relu(lin(x, w1, b1)), w2, b2)), w3, b3).squeeze(1)
    qq = torch.tensor(q, dtype=torch.float64)
    qt = qq[torch.arange(q.shape[0]), torch.tensor(batch["actions"], dtype=torch.int64)]
    d = qt - v
    wgt = torch.where(d >= 0, torch.full_like(d, tau), torch.full_like(d, 1 - tau))
    loss = (wgt * d * d).mean()
    opt.zero_grad()
    loss.backward()
    g0 = t.grad.detach().clone()
    n0 = float(torch.linalg.vector_norm(g0))
    torch.nn.utils.clip_grad_norm_([t], max_norm=0.70 * w.max_grad_norm)
    total = t.grad.detach().clone()
    for k, src in enumerate(aux if aux is not None else []):
        holder = torch.zeros_like(t, requires_grad=True)
        holder.grad = torch.tensor(src, dtype=torch.float64)
        torch.nn.utils.clip_grad_norm_([holder], max_norm=w.budget[k + 1] * w.max_grad_norm)
        total += holder.grad
    t.grad = total
    torch.nn.utils.clip_grad_norm_([t], max_norm=w.max_grad_norm)
    opt.step()
    adv = torch.clamp(qq - v.detach()[:, None], -10, 10)
    pi = torch.softmax(w.beta * adv, dim=1)
    return float(loss.detach()), v.detach().numpy(), pi.numpy(), g0.numpy(), n0


def _run(w, steps, with_aux):
    rep = synth.make_replay(w)
    cfg = step.config_from_workload(w)
    nets = [step.NetState.fresh(synth.make_params(w, k), w.taus[k]) for k in range(w.n_nets)]
    tparams = [torch.tensor(synth.make_params(w, k), dtype=torch.float64, requires_grad=True)
               for k in range(w.n_nets)]
    opts = [torch.optim.AdamW([tp], lr=w.lr, betas=(w.beta1, w.beta2), eps=w.eps,
                              weight_decay=w.weight_decay) for tp in tparams]
    for st in range(steps):
        q = synth.make_q(w, st)
        aux = [synth.make_aux(w, st, k) for k in range(w.n_nets)] if with_aux else None
        out = step.train_step(cfg, rep, st, q, nets, aux)
        for k in range(w.n_nets):
            loss, v, pi, g0, n0 = _torch_step(w, tparams[k], opts[k], out["batch"], q, w.taus[k],
                                              aux[k] if aux else None)
            # the two sides drift apart by the +1e-6 in torch's clip scale:
            # ~1e-9 in the weights per step, hence the tolerances
            assert abs(out["loss"][k] - loss) <= 1e-8 * abs(loss)
            np.testing.assert_allclose(out["v"][k], v, rtol=1e-7, atol=1e-9)
            np.testing.assert_allclose(out["pi"][k], pi, rtol=1e-7, atol=1e-12)
            np.testing.assert_allclose(out["grad"][k], g0, rtol=1e-6, atol=1e-10)
            assert abs(out["norms"][k][0] - n0) <= 1e-7 * n0
            np.testing.assert_allclose(nets[k].params, tparams[k].detach().numpy(), rtol=0,
                                       atol=2e-9 * (st + 1))
        assert out["norms"][0][4] <= w.max_grad_norm * (1 + 1e-12)


def test_tiny_step_matches_torch():
    _run(synth.TINY, 3, with_aux=False)


def test_twin_step_matches_torch():
    w = dataclasses.replace(synth.TWIN, batch=200, capacity=4096, hidden=32, prec="fp32")
    _run(w, 2, with_aux=False)


def test_budgeted_step_matches_torch():
    w = dataclasses.replace(synth.BUDGETED, batch=128, capacity=2048, hidden=24)
    _run(w, 3, with_aux=True)


def test_her_rows_are_last_in_step_batch():
    w = synth.TINY
    rep = synth.make_replay(w)
    cfg = step.config_from_workload(w)
    nets = [step.NetState.fresh(synth.make_params(w), 0.7)]
    out = step.train_step(cfg, rep, 0, synth.make_q(w, 0), nets)
    donor = out["batch"]["donor_idx"]
    n_her = her.her_count(w.batch, w.her_ratio)
    assert (donor[: w.batch - n_her] == -1).all() and (donor[w.batch - n_her:] >= 0).all()
