"""tt_weighted_logprob against the oracle (branch-average == weighted-token loss)."""
import numpy as np
import pytest
import torch

import synth
from oracle import logprob as L
from oracle import tree as T
from tests._util import DLOGIT_ATOL, DLOGIT_RTOL, LOGP_ATOL, f64, to_dev_bf16

pytestmark = pytest.mark.gpu


def _run(tt, bits, targets, weights, g=1.0, want=True, ld=None):
    z = to_dev_bf16(bits)
    if ld is not None:  # rows ld elements apart (a padded buffer, the vectorised kernels' layout for any V)
        zp = torch.full((z.shape[0], ld), float("nan"), dtype=torch.bfloat16, device="cuda")
        zp[:, :z.shape[1]] = z
        z = zp[:, :z.shape[1]]
    y = torch.tensor(targets, dtype=torch.int32, device="cuda")
    w = None if weights is None else torch.tensor(weights, dtype=torch.float32, device="cuda")
    err = tt.new_err("cuda")
    logp, loss, dl = tt.weighted_logprob(z, y, w, g=g, want_dlogits=want, err=err)
    torch.cuda.synchronize()
    return logp.cpu().numpy(), float(loss.item()), (None if dl is None else dl.float().cpu().numpy()), int(err.item())


def _check_dlogits(dl, ref):
    bad = np.abs(dl - ref) > DLOGIT_RTOL * np.abs(ref) + DLOGIT_ATOL
    assert not bad.any(), f"{bad.sum()} dlogits outside tolerance; worst {np.abs(dl - ref)[bad].max()}"


def test_tiny_workload_vs_branch_average(tt):
    inp = synth.logprob_inputs(0)
    tt_ = T.tables(inp["tree"].seg_parent, inp["tree"].seg_len)
    w = tt_.tok_weight                                   # fp32 branch fractions, as the GPU receives
    z = f64(inp["logits"])
    lp_ref, loss_ref, dl_ref = L.weighted_token_loss(z, inp["targets"], w)
    _, loss_branch, _ = L.branch_average_loss(tt_, z, inp["targets"])
    assert abs(loss_branch - loss_ref) < 1e-3          # fp32 weights vs exact fractions
    logp, loss, dl, err = _run(tt, inp["logits"], inp["targets"], w)
    assert err == 0
    assert np.abs(logp - lp_ref).max() <= LOGP_ATOL
    assert abs(loss - loss_ref) <= LOGP_ATOL
    _check_dlogits(dl, dl_ref)


@pytest.mark.parametrize("N,V,g", [(1, 1, 1.0), (3, 7, 0.5), (37, 1000, 1.0), (64, 2049, 2.0), (17, 30011, 1.0),
                                   (9, 163840, 1.0), (5, 200003, 1.0), (40, 1001, 1.0)])
def test_shapes(tt, N, V, g):
    rng = np.random.default_rng(N * 7 + V)
    bits = synth.normal_bf16(rng, (N, V), 2.0)
    y = rng.integers(0, V, N).astype(np.int32)
    w = rng.random(N).astype(np.float32)
    lp_ref, loss_ref, dl_ref = L.weighted_token_loss(f64(bits), y, w, g=g)
    logp, loss, dl, err = _run(tt, bits, y, w, g=g)
    assert err == 0
    assert np.abs(logp - lp_ref).max() <= LOGP_ATOL
    assert abs(loss - loss_ref) <= LOGP_ATOL
    _check_dlogits(dl, dl_ref)
    # forward only, no weights (= 1)
    logp2, loss2, dl2, err2 = _run(tt, bits, y, None, want=False)
    assert dl2 is None and err2 == 0
    np.testing.assert_array_equal(logp2, logp)
    assert abs(loss2 - float(-(lp_ref).sum())) <= LOGP_ATOL * max(1, N / 100)


def test_extreme_logits(tt):
    # one dominant logit per row, -inf-free but huge spread; uniform rows
    N, V = 6, 4096
    z = np.zeros((N, V), np.float32)
    z[0, 17] = 80.0
    z[1] = np.linspace(-60, 60, V)
    z[2] = 3.0
    z[3, ::2] = -100.0
    z[4] = -30.0
    z[4, 5] = 30.0
    z[5] = np.random.default_rng(0).standard_normal(V) * 10
    bits = synth.f32_to_bf16_bits(z)
    y = np.array([17, 0, 5, 1, 5, 100], np.int32)
    w = np.ones(N, np.float32)
    lp_ref, loss_ref, dl_ref = L.weighted_token_loss(f64(bits), y, w)
    logp, loss, dl, err = _run(tt, bits, y, w)
    assert err == 0
    assert np.abs(logp - lp_ref).max() <= LOGP_ATOL
    assert logp[2] == pytest.approx(-np.log(V), abs=1e-5)
    _check_dlogits(dl, dl_ref)


def test_invalid_target(tt):
    rng = np.random.default_rng(1)
    bits = synth.normal_bf16(rng, (4, 100), 1.0)
    logp, loss, dl, err = _run(tt, bits, np.array([3, 100, -1, 5], np.int32), np.ones(4, np.float32))
    assert err == -1
    assert np.isnan(logp[1]) and np.isnan(logp[2]) and np.isfinite(logp[0]) and np.isnan(loss)


def test_full_vocab_workload(tt):
    """Config 2 at full size: all rows' logp and the loss; dlogits on sampled rows."""
    inp = synth.logprob_inputs(2)
    tt_ = T.tables(inp["tree"].seg_parent, inp["tree"].seg_len)
    bits, y, w = inp["logits"], inp["targets"], tt_.tok_weight
    err = tt.new_err("cuda")
    logp_d, loss_d, dl_d = tt.weighted_logprob(to_dev_bf16(bits), torch.tensor(y, device="cuda"),
                                               torch.tensor(w, device="cuda"), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    logp, loss = logp_d.cpu().numpy(), float(loss_d.item())
    lp_ref, loss_ref = L.weighted_loss_sampled(lambda lo, hi: f64(bits[lo:hi]), bits.shape[0], y, w)
    assert np.abs(logp - lp_ref).max() <= LOGP_ATOL
    assert abs(loss - loss_ref) <= LOGP_ATOL, (loss, loss_ref)
    rows = np.unique(np.r_[0, 1, bits.shape[0] - 1, np.random.default_rng(0).integers(0, bits.shape[0], 24)])
    _, _, dl_ref = L.weighted_token_loss(f64(bits[rows]), y[rows], w[rows])
    dl = dl_d[torch.tensor(rows, device="cuda")].float().cpu().numpy()
    _check_dlogits(dl, dl_ref)


def test_rescale_factors_closed_form(tt):
    """Rows where every logit but one equals −a: every thread's, warp's and CTA's partial sum is rescaled to the row
    maximum by exp(−a), so the accuracy of the kernel's rescaling exponential (a Cody–Waite reduction and a fitted
    polynomial, ≈2e-9 relative) decides logp. Against the closed form logp = z_y − log(1 + (V − 1)·e^(−a)) in fp64,
    at 2e-6 (about two fp32 ulps of logp), for a over [0.25, 11] (beyond, the rescaled terms stop mattering), with
    the maximum placed in different CTAs of the cluster and the target on or off it."""
    V = 151936
    avals = [0.25, 0.5, 1.0, 1.5, 2.5, 3.0, 4.25, 5.0, 6.5, 7.25, 8.0, 9.0, 10.5, 11.0]
    N = len(avals)
    rng = np.random.default_rng(5)
    z = np.empty((N, V), np.float32)
    pmax = rng.integers(0, V, N)
    for i, a in enumerate(avals):
        z[i] = -a
        z[i, pmax[i]] = 0.0
    bits = synth.f32_to_bf16_bits(z)
    assert np.array_equal(synth.bf16_bits_to_f32(bits), z)  # the values are bf16-exact
    y = np.where(np.arange(N) % 2 == 0, pmax, (pmax + 1 + rng.integers(0, V - 1, N)) % V).astype(np.int32)
    logp, _, _, err = _run(tt, bits, y, None, want=False)
    assert err == 0
    a = np.asarray(avals, np.float64)
    zy = np.where(y == pmax, 0.0, -a)
    ref = zy - np.log1p((V - 1) * np.exp(-a))
    assert np.abs(logp - ref).max() <= 2e-6, np.abs(logp - ref)


def _logprob_launches(tt, bits, y, w, ld=None):
    """Run once with launch timing on; returns (logp, loss, dlogits, err, launches of the log-prob class)."""
    tt.kernel_timing(True)
    out = _run(tt, bits, y, w, ld=ld)
    tt.kernel_timing(False)
    times, _ = tt.kernel_timing_read()
    return out + (times["logprob"][1],)


def _idle_sm_case(n, V, tail):
    """n rows at V whose last len(tail) rows are `tail` (float32 rows): the rows the idle SMs take."""
    rng = np.random.default_rng(n + V)
    z = (rng.standard_normal((n, V)) * 2.0).astype(np.float32)
    z[n - len(tail):] = tail
    return synth.f32_to_bf16_bits(z), rng


def test_idle_sm_rows(tt):
    """Batches of at least four rows per SM at a vocabulary that needs clusters of 8 CTAs: the clusters take the
    first rows and a row kernel on the SMs they leave idle takes the last ones (on a 152-SM GB300 the 36 clusters
    leave 8 SMs idle: the last 22 of 700 rows). Every logp, the loss and the dlogits of rows on both sides of the
    split against the oracle, at V = 151939 (a ragged tail of 3 elements), with extreme rows (a dominant logit, a
    ±60 ramp, uniform, −100 on every other element, the maximum in the ragged tail) and an invalid target among the
    last rows; repeat calls bitwise equal."""
    n, V = 700, 151939
    tail = np.zeros((6, V), np.float32)
    tail[0, 17] = 80.0
    tail[1] = np.linspace(-60, 60, V)
    tail[2] = 3.0
    tail[3, ::2] = -100.0
    tail[4] = -30.0
    tail[4, 5] = 30.0
    tail[5, -1] = 9.0  # the maximum in the ragged tail
    bits, rng = _idle_sm_case(n, V, tail)
    y = rng.integers(0, V, n).astype(np.int32)
    y[n - 6:] = [17, 0, 5, 1, 5, V - 1]
    w = rng.random(n).astype(np.float32)
    ld = (V + 7) // 8 * 8  # rows padded to whole 16-byte vectors (NaN padding, never read)
    logp, loss, dl, err, launches = _logprob_launches(tt, bits, y, w, ld=ld)
    assert err == 0
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert launches == 2  # the cluster kernel and the row kernel
    lp_ref, loss_ref = L.weighted_loss_sampled(lambda lo, hi: f64(bits[lo:hi]), n, y, w)
    assert np.abs(logp - lp_ref).max() <= LOGP_ATOL
    assert abs(loss - loss_ref) <= LOGP_ATOL * max(1.0, n / 100)
    rows = np.r_[0, 1, 300, n - 30, n - 23, n - 22, n - 21, n - 12, np.arange(n - 6, n)]
    _, _, dl_ref = L.weighted_token_loss(f64(bits[rows]), y[rows], w[rows])
    _check_dlogits(dl[rows], dl_ref)
    again = _run(tt, bits, y, w, ld=ld)
    np.testing.assert_array_equal(again[0], logp)
    np.testing.assert_array_equal(again[2], dl)
    y[n - 1] = V  # invalid target on the row kernel's side
    logp3, loss3, _, err3 = _run(tt, bits, y, w, ld=ld)
    assert err3 == -1 and np.isnan(logp3[n - 1]) and np.isnan(loss3)
    assert np.abs(logp3[:n - 1] - lp_ref[:n - 1]).max() <= LOGP_ATOL


def test_idle_sm_rows_rescale_closed_form(tt):
    """The closed-form rows of test_rescale_factors_closed_form placed last in a 700-row batch at V = 151936, so that
    the row kernel on the idle SMs computes them: the same 2e-6 bound."""
    V = 151936
    avals = [0.25, 0.5, 1.0, 2.5, 4.25, 6.5, 8.0, 9.0, 10.5, 11.0]
    rng = np.random.default_rng(6)
    tail = np.empty((len(avals), V), np.float32)
    pmax = rng.integers(0, V, len(avals))
    for i, a in enumerate(avals):
        tail[i] = -a
        tail[i, pmax[i]] = 0.0
    n = 700
    bits, rng2 = _idle_sm_case(n, V, tail)
    y = rng2.integers(0, V, n).astype(np.int32)
    yt = np.where(np.arange(len(avals)) % 2 == 0, pmax, (pmax + 1 + rng.integers(0, V - 1, len(avals))) % V)
    y[n - len(avals):] = yt
    logp, _, _, err = _run(tt, bits, y, None, want=False)
    assert err == 0
    a = np.asarray(avals, np.float64)
    ref = np.where(yt == pmax, 0.0, -a) - np.log1p((V - 1) * np.exp(-a))
    assert np.abs(logp[n - len(avals):] - ref).max() <= 2e-6, np.abs(logp[n - len(avals):] - ref)
