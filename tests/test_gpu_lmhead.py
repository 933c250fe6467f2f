"""tt_lmhead_logprob (LM head z = H·Wᵀ fused with the weighted log-prob) against the oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import lmhead as LH
from tests._util import GRAD_RL2, LOGP_ATOL, dev_to_f64, f64, rel_l2, to_dev_bf16

# The loss is a weighted sum of per-row log-probabilities whose logits come
# from an fp32-accumulated bf16 product: 1e-4 per unit of total weight (the
# per-token mean loss within 1e-4).
def loss_atol(w):
    return LOGP_ATOL * max(1.0, float(np.sum(w)))

pytestmark = pytest.mark.gpu


def _run(tt, H, W, y, w, ws=None):
    err = tt.new_err("cuda")
    yt = torch.tensor(y, dtype=torch.int32, device="cuda")
    wt = None if w is None else torch.tensor(w, dtype=torch.float32, device="cuda")
    logp, lse, loss = tt.lmhead_logprob(H, W, yt, wt, err=err, ws=ws)
    torch.cuda.synchronize()
    return logp.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), float(loss.item()), \
        int(err.item())


# several 128-row and 256-column tiles with ragged tails, one tile, K of one and several 64-wide steps
@pytest.mark.parametrize("N,V,Hd", [(1, 1, 64), (77, 1000, 64), (300, 3001, 128), (129, 256, 192),
                                    (513, 4099, 256), (256, 511, 64)])
def test_shapes_vs_oracle(tt, N, V, Hd):
    d = synth.lmhead_inputs(N + V + Hd, n_rows=N, vocab=V, hidden=Hd)
    rng = np.random.default_rng(N)
    w = rng.random(N).astype(np.float32)
    ref = LH.lmhead_weighted_loss(f64(d["H"]), f64(d["W"]), d["targets"], w.astype(np.float64), want_grads=False)
    logp, lse, loss, err = _run(tt, to_dev_bf16(d["H"]), to_dev_bf16(d["W"]), d["targets"], w)
    assert err == 0
    assert np.abs(logp - ref["logp"]).max() <= LOGP_ATOL
    assert np.abs(lse - ref["lse"]).max() <= LOGP_ATOL
    assert abs(loss - ref["loss"]) <= loss_atol(w), (loss, ref["loss"])
    # no weights = all ones; the same per-row values
    logp1, lse1, loss1, err1 = _run(tt, to_dev_bf16(d["H"]), to_dev_bf16(d["W"]), d["targets"], None)
    assert err1 == 0
    np.testing.assert_array_equal(logp1, logp)
    assert abs(loss1 + logp1.sum()) <= 1e-9 * max(1.0, abs(loss1))


def test_matches_the_unfused_log_prob_call(tt):
    """The fused call equals tt_weighted_logprob on the bf16-rounded logits up to that rounding."""
    d = synth.lmhead_inputs(5, n_rows=200, vocab=5000, hidden=128)
    H, W = to_dev_bf16(d["H"]), to_dev_bf16(d["W"])
    y = torch.tensor(d["targets"], dtype=torch.int32, device="cuda")
    logp, lse, loss = tt.lmhead_logprob(H, W, y)
    z = (H.float() @ W.float().T).to(torch.bfloat16)
    logp2, loss2, _ = tt.weighted_logprob(z, y, want_dlogits=False)
    torch.cuda.synchronize()
    # bf16 rounding of z (|z| <~ 10, half an ulp <= 2^-5) moves logp by at most ~2·2^-5
    assert (logp - logp2).abs().max().item() <= 0.07


def test_invalid_target_sets_error_and_nan(tt):
    d = synth.lmhead_inputs(9, n_rows=40, vocab=700, hidden=64)
    y = d["targets"].copy()
    y[5] = 700
    logp, lse, loss, err = _run(tt, to_dev_bf16(d["H"]), to_dev_bf16(d["W"]), y, None)
    assert err == -1
    assert np.isnan(logp[5]) and np.isnan(loss)
    ok = np.arange(40) != 5
    ref = LH.lmhead_weighted_loss(f64(d["H"]), f64(d["W"]), np.where(ok, y, 0), np.ones(40), want_grads=False)
    assert np.abs(logp[ok] - ref["logp"][ok]).max() <= LOGP_ATOL


def test_argument_errors(tt):
    H = torch.zeros(16, 96, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(tt.TTError) as e:
        tt.lmhead_logprob(H, H, y)  # Hd = 96 is not a multiple of 64
    assert e.value.code == -3
    H = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tt.TTError) as e:
        tt.lmhead_logprob(H, H, y, ws=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -4


def test_repeatable_bitwise(tt):
    d = synth.lmhead_inputs(3, n_rows=333, vocab=9000, hidden=128)
    H, W = to_dev_bf16(d["H"]), to_dev_bf16(d["W"])
    y = torch.tensor(d["targets"], dtype=torch.int32, device="cuda")
    a = tt.lmhead_logprob(H, W, y)
    b = tt.lmhead_logprob(H, W, y)
    torch.cuda.synchronize()
    for x, z in zip(a, b):
        assert torch.equal(x, z)


def test_full_size_sampled_rows(tt):
    """The benchmarked shape (config 2's tree, Qwen3-1.7B hidden 2048, V = 151936, the launch bench.py times):
    sampled rows against the oracle, the loss against −Σ w·logp of the returned rows."""
    d = synth.lmhead_inputs(0)
    N = d["H"].shape[0]
    H, W = to_dev_bf16(d["H"]), to_dev_bf16(d["W"])
    rng = np.random.default_rng(1)
    w = rng.random(N).astype(np.float32)
    y = torch.tensor(d["targets"], dtype=torch.int32, device="cuda")
    err = tt.new_err("cuda")
    logp, lse, loss = tt.lmhead_logprob(H, W, y, torch.tensor(w, device="cuda"), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    logp = logp.cpu().numpy().astype(np.float64)
    rows = np.r_[0, 1, 127, 128, 4097, N - 129, N - 1]
    lse_ref, logp_ref = LH.lmhead_rows(f64(d["H"][rows]), d["W"], d["targets"][rows], np.arange(len(rows)),
                                       widen=f64)
    assert np.abs(logp[rows] - logp_ref).max() <= LOGP_ATOL
    assert np.abs(lse.cpu().numpy()[rows] - lse_ref).max() <= LOGP_ATOL
    assert np.isfinite(logp).all() and (logp < 0).all()
    assert abs(float(loss.item()) + (w.astype(np.float64) * logp).sum()) <= 1e-6 * abs(float(loss.item()))


@pytest.mark.parametrize("N,V,Hd,g", [(77, 1000, 64, 1.0), (300, 3001, 128, 0.5), (129, 256, 192, 2.0),
                                      (513, 4099, 256, 1.0)])
def test_backward_vs_oracle(tt, N, V, Hd, g):
    """dH = dz·W and dW = dzᵀ·H (dz = g·w·(softmax − onehot)) against the fp64 oracle: relative L2 1e-2, as for
    the attention gradients (bf16 inputs and dz, fp32 accumulation)."""
    d = synth.lmhead_inputs(7 * N + V, n_rows=N, vocab=V, hidden=Hd)
    w = np.random.default_rng(N + 1).random(N).astype(np.float32)
    ref = LH.lmhead_weighted_loss(f64(d["H"]), f64(d["W"]), d["targets"], w.astype(np.float64), g=g)
    H, W = to_dev_bf16(d["H"]), to_dev_bf16(d["W"])
    y = torch.tensor(d["targets"], dtype=torch.int32, device="cuda")
    wt = torch.tensor(w, device="cuda")
    err = tt.new_err("cuda")
    logp, lse, loss = tt.lmhead_logprob(H, W, y, wt, err=err)
    dh, dw = tt.lmhead_logprob_bwd(H, W, y, lse, wt, g=g, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert rel_l2(dev_to_f64(dh), ref["dH"]) <= GRAD_RL2
    assert rel_l2(dw.cpu().numpy(), ref["dW"]) <= GRAD_RL2
    # bitwise repeatable
    dh2, dw2 = tt.lmhead_logprob_bwd(H, W, y, lse, wt, g=g)
    torch.cuda.synchronize()
    assert torch.equal(dh, dh2) and torch.equal(dw, dw2)


def test_backward_full_size_sampled_rows_and_column_sums(tt):
    """The benchmarked shape: dH on sampled rows against the oracle (dz row by row in fp64, W in vocabulary chunks),
    and the property Σ_v dW[v] = Σ_t (Σ_v dz_tv) H_t = 0 (every row of dz sums to g·w·(1 − 1))."""
    d = synth.lmhead_inputs(0)
    N = d["H"].shape[0]
    H, W = to_dev_bf16(d["H"]), to_dev_bf16(d["W"])
    w = np.random.default_rng(1).random(N).astype(np.float32)
    y = torch.tensor(d["targets"], dtype=torch.int32, device="cuda")
    wt = torch.tensor(w, device="cuda")
    err = tt.new_err("cuda")
    logp, lse, loss = tt.lmhead_logprob(H, W, y, wt, err=err)
    dh, dw = tt.lmhead_logprob_bwd(H, W, y, lse, wt, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = np.r_[0, 127, 4097, N - 1]
    Hs = f64(d["H"][rows])
    # oracle dH rows: dz_t = w_t (softmax_t − onehot), dH_t = dz_t · W, with W widened chunk by chunk
    lse_ref, _ = LH.lmhead_rows(Hs, d["W"], d["targets"][rows], np.arange(len(rows)), widen=f64)
    dh_ref = np.zeros((len(rows), d["Hd"]))
    for lo in range(0, d["V"], 16384):
        Wc = f64(d["W"][lo:lo + 16384])
        p = np.exp(Hs @ Wc.T - lse_ref[:, None])
        inside = (d["targets"][rows] >= lo) & (d["targets"][rows] < lo + len(Wc))
        p[inside, d["targets"][rows][inside] - lo] -= 1.0
        dh_ref += (w[rows, None] * p) @ Wc
    assert rel_l2(dev_to_f64(dh)[rows], dh_ref) <= GRAD_RL2
    col = dw.double().sum(0).cpu().numpy()
    assert np.abs(col).max() <= 1e-3 * dw.double().abs().sum(0).max().item()
