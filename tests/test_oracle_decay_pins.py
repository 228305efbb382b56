"""The fp64 oracle of the tau-decay cell against facts other than itself (CPU only).

Each pin is chosen so that a plausible mistake in the oracle fails it:
  * central finite differences on every gradient entry (a wrong sign, factor or index in the
    hand-written backward, including dtau);
  * tau -> 0: the decay underflows to 0 and the cell is exactly a tanh RNN, compared with
    torch.nn.RNN and its autograd gradients (the (1 - d) / d roles, W_in / W_rec order);
  * ts = 0: no decay at all, h stays h0, every gradient but dh0 vanishes and dh0 = sum_t dH;
  * W = 0, b = 0: h_t = h0 exp(-S_t / tau) with S_t the running sum of ts, in closed form, and
    so are dh0 and dtau (the direction ts / tau of the exponent and the dtau formula);
  * the batch gradient is the sum of the per-row gradients.
"""
import numpy as np
import pytest

import oracle.decay as decay
from recurrent_cfc_cell_gb300 import inputs


@pytest.fixture(scope="module")
def lib():
    return decay.default()


def _rel(x, y) -> float:
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    return float(np.max(np.abs(x - y)) / max(np.max(np.abs(y)), 1e-300))


def _case(B=2, K=3, n_x=2, C=3, seed=3, **kw) -> dict:
    inp = inputs.make_decay_inputs(inputs.decay_custom(B, K, n_x, C, seed=seed, **kw))
    return {k: v.astype(np.float64) for k, v in inp.items()}


def test_finite_differences(lib):
    inp = _case()
    g = lib.backward(inp)
    h = 1e-5
    names = {"W": "dW", "b": "db", "tau": "dtau", "x": "dx", "h0": "dh0"}
    for p, gname in names.items():
        fd = np.zeros_like(inp[p])
        flat = inp[p].reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + h
            lp = lib.loss(inp)
            flat[i] = keep - h
            lm = lib.loss(inp)
            flat[i] = keep
            fd.reshape(-1)[i] = (lp - lm) / (2 * h)
        assert _rel(g[gname], fd) <= 1e-6, (p, _rel(g[gname], fd))


def test_tau_to_zero_is_a_tanh_rnn(lib):
    torch = pytest.importorskip("torch")
    B, K, n_x, C = 3, 5, 4, 6
    inp = _case(B, K, n_x, C, seed=5)
    inp["tau"][:] = 1e-4  # ts >= 0.5: exp(-5000) is 0 in fp64
    o = lib.step(inp)
    rnn = torch.nn.RNN(n_x, C, nonlinearity="tanh", bias=True).double()
    with torch.no_grad():
        rnn.weight_ih_l0.copy_(torch.from_numpy(inp["W"][:, :n_x]))
        rnn.weight_hh_l0.copy_(torch.from_numpy(inp["W"][:, n_x:]))
        rnn.bias_ih_l0.copy_(torch.from_numpy(inp["b"]))
        rnn.bias_hh_l0.zero_()
    x = torch.from_numpy(inp["x"]).requires_grad_(True)
    h0 = torch.from_numpy(inp["h0"])[None].clone().requires_grad_(True)
    H, _ = rnn(x, h0)
    (H * torch.from_numpy(inp["dH"])).sum().backward()
    assert _rel(o["H"], H.detach().numpy()) <= 1e-13
    dW = np.concatenate([rnn.weight_ih_l0.grad.numpy(), rnn.weight_hh_l0.grad.numpy()], axis=1)
    assert _rel(o["dW"], dW) <= 1e-12
    assert _rel(o["db"], rnn.bias_ih_l0.grad.numpy()) <= 1e-12
    assert _rel(o["dx"], x.grad.numpy()) <= 1e-12
    assert _rel(o["dh0"], h0.grad.numpy()[0]) <= 1e-12
    assert np.max(np.abs(o["dtau"])) == 0.0


def test_no_time_step_keeps_the_state(lib):
    inp = _case(B=3, K=4, n_x=3, C=5, seed=7)
    inp["ts"][:] = 0.0
    o = lib.step(inp)
    for t in range(4):
        assert np.array_equal(o["H"][t], inp["h0"])
    for k in ("dW", "db", "dtau", "dx", "da"):
        assert np.max(np.abs(o[k])) == 0.0, k
    assert _rel(o["dh0"], inp["dH"].sum(axis=0)) <= 1e-15


def test_pure_decay_closed_form(lib):
    inp = _case(B=3, K=6, n_x=2, C=4, seed=9)
    inp["W"][:] = 0.0
    inp["b"][:] = 0.0
    o = lib.step(inp)
    S = np.cumsum(inp["ts"], axis=0)                      # S_t = ts_0 + ... + ts_t, [K, B]
    tau = inp["tau"]
    H = inp["h0"][None] * np.exp(-S[..., None] / tau)     # [K, B, C]
    assert _rel(o["H"], H) <= 1e-14
    dh0 = (inp["dH"] * np.exp(-S[..., None] / tau)).sum(axis=0)
    assert _rel(o["dh0"], dh0) <= 1e-14
    # dh_t/dtau = h_t S_t / tau^2 for every (t, b, i)
    dtau = (inp["dH"] * H * S[..., None] / tau ** 2).sum(axis=(0, 1))
    assert _rel(o["dtau"], dtau) <= 1e-13


def test_batch_gradient_is_the_sum_of_rows(lib):
    inp = _case(B=4, K=5, n_x=3, C=4, seed=13)
    full = lib.step(inp)
    acc = {k: 0.0 for k in ("dW", "db", "dtau")}
    for b in range(4):
        one = dict(inp, x=inp["x"][:, b:b + 1], h0=inp["h0"][b:b + 1], ts=inp["ts"][:, b:b + 1],
                   dH=inp["dH"][:, b:b + 1])
        o = lib.step(one)
        for k in acc:
            acc[k] = acc[k] + o[k]
        assert _rel(o["H"][:, 0], full["H"][:, b]) <= 1e-15
        assert _rel(o["dx"][:, 0], full["dx"][:, b]) <= 1e-14
        assert _rel(o["dh0"][0], full["dh0"][b]) <= 1e-14
    for k, v in acc.items():
        assert _rel(v, full[k]) <= 1e-13, k
