"""Pins for the CPU oracle: checks that do not restate its formulas.

Each test ties the oracle to something fixed outside it -- a value printed on
one of the transcript pages (tests/golden/page_examples.json), a closed form,
an invariant of the epilogue, brute force written independently here, or a
library routine (PyTorch CPU ops in fp64) on a special case.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


def rand_case(rng, N, Cin, Cout, D, H, W, k, bias=True):
    x = rng.standard_normal((N, Cin, D, H, W)).astype(np.float32)
    w = (rng.uniform(-1, 1, (Cin, Cout, k, k, k)) / math.sqrt(Cout * k ** 3)).astype(np.float32)
    b = rng.uniform(-0.3, 0.3, Cout).astype(np.float32) if bias else None
    return x, w, b


# ---------------------------------------------------------------- shapes ----

@pytest.mark.parametrize("case", GOLDEN["shapes"], ids=lambda c: c["page"].split()[0])
def test_output_shape_matches_pages(case):
    N, Cin, D, H, W = case["x"]
    dims = [oracle.output_size(v, case["k"], case["stride"], case["pad"], case["out_pad"])
            for v in (D, H, W)]
    assert [N, case["Cout"], *dims] == case["y"]


def test_groupnorm_group_size_from_page():
    g = GOLDEN["groupnorm_elements_per_group"]
    D = oracle.output_size(g["x"][2], g["k"], 1, 0, 0)
    assert (g["Cout"] // g["groups"]) * D ** 3 == g["value"]


def test_product_count_printed_on_page():
    g = GOLDEN["scatter_product_count"]
    N, Cin, D, H, W = g["x"]
    in_range, total = oracle.count_products(N, Cin, g["Cout"], D, H, W, g["k"], g["stride"],
                                            g["pad"], g["out_pad"])
    assert total == g["value"]
    assert 0 < in_range < total


def test_product_count_in_range_brute_force():
    # independent enumeration of (i, t) pairs landing inside the output, per dimension
    N, Cin, Cout, D, H, W, k, s, p, op = 2, 3, 2, 4, 5, 3, 3, 2, 1, 1
    Do, Ho, Wo = (oracle.output_size(v, k, s, p, op) for v in (D, H, W))
    hits = 0
    for i_d in range(D):
        for i_h in range(H):
            for i_w in range(W):
                for td in range(k):
                    for th in range(k):
                        for tw in range(k):
                            o = (i_d * s - p + td, i_h * s - p + th, i_w * s - p + tw)
                            if all(0 <= a < b for a, b in zip(o, (Do, Ho, Wo))):
                                hits += 1
    in_range, total = oracle.count_products(N, Cin, Cout, D, H, W, k, s, p, op)
    assert in_range == hits * N * Cin * Cout
    assert total == N * Cin * Cout * D * H * W * k ** 3


# ------------------------------------------------- 1-D examples in 3-D ----

def _line_response(axis, in_len, k, s, p, op, i, t):
    """Oracle output for a unit input at position i along `axis` and a weight that is
    one-hot at tap t along `axis`.  Along the other two axes the input has length 1
    and the tap is p, which places the value at output index 0 there."""
    shape = [1, 1, 1]
    shape[axis] = in_len
    x = np.zeros((1, 1, *shape), np.float32)
    idx = [0, 0, 0]
    idx[axis] = i
    x[(0, 0, *idx)] = 1.0
    w = np.zeros((1, 1, k, k, k), np.float32)
    tap = [p, p, p]
    tap[axis] = t
    w[(0, 0, *tap)] = 1.0
    Y = oracle.convt3d_scatter(x, w, None, stride=s, pad=p, out_pad=op)
    return Y[0, 0]


def _collect_terms(axis, in_len, k, s, p, op):
    """For each output index along `axis`, the (i, t) pairs that reach it."""
    out_len = oracle.output_size(in_len, k, s, p, op)
    terms = {o: [] for o in range(out_len)}
    for i in range(in_len):
        for t in range(k):
            R = _line_response(axis, in_len, k, s, p, op, i, t)
            for pos in np.argwhere(R != 0):
                pos = tuple(int(v) for v in pos)
                assert all(pos[a] == 0 for a in range(3) if a != axis)
                assert R[pos] == 1.0
                terms[pos[axis]].append((i, t))
    return terms


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_one_d_matrix_example(axis):
    g = GOLDEN["one_d_matrix_example"]
    terms = _collect_terms(axis, g["in_len"], g["k"], g["stride"], g["pad"], 0)
    expect = [sorted(tuple(p) for p in row) for row in g["terms"]]
    assert [sorted(terms[o]) for o in range(len(expect))] == expect
    assert len(terms) == len(expect)


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_one_d_impulse(axis):
    g = GOLDEN["one_d_impulse"]
    k = g["k"]
    kern = np.array([3.0, 5.0, 7.0], np.float32)  # k0, k1, k2
    shape = [1, 1, 1]
    shape[axis] = len(g["input"])
    x = np.zeros((1, 1, *shape), np.float32)
    for i, v in enumerate(g["input"]):
        idx = [0, 0, 0]
        idx[axis] = i
        x[(0, 0, *idx)] = v
    w = np.zeros((1, 1, k, k, k), np.float32)
    for t in range(k):
        tap = [0, 0, 0]
        tap[axis] = t
        w[(0, 0, *tap)] = kern[t]
    Y = oracle.convt3d_scatter(x, w, None, stride=g["stride"], pad=g["pad"])[0, 0]
    line = np.moveaxis(Y, axis, 0)[:, 0, 0]
    expect = [0.0 if t is None else float(kern[t]) for t in g["out_tap"]]
    assert line.tolist() == expect
    # the other two axes: only index 0 is non-zero
    rest = np.moveaxis(Y, axis, 0)[:, 1:, :]
    assert not rest.any()


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_stride2_tap_table(axis):
    g = GOLDEN["stride2_tap_table"]
    terms = _collect_terms(axis, g["in_len"], g["k"], g["stride"], g["pad"], g["out_pad"])
    for o, pairs in g["rows"].items():
        assert sorted(terms[int(o)]) == sorted(tuple(p) for p in pairs)
    lo, hi = g["alternation_rows"]
    for o in range(lo, hi):  # the page's 1, 2, 1, 2 pattern below the top edge
        assert len(terms[o]) == (1 if o % 2 == 0 else 2)


# ------------------------------------ stride-1 flipped-kernel identity ----

def _flipped_correlation(x, w, pad_eff):
    """Independent gather form: zero-pad x by pad_eff, correlate with the kernel
    flipped in all three spatial axes and with in/out channels swapped."""
    N, Cin, D, H, W = x.shape
    k = w.shape[2]
    wf = np.flip(np.transpose(w.astype(np.float64), (1, 0, 2, 3, 4)), axis=(2, 3, 4))
    xp = np.pad(x.astype(np.float64), ((0, 0), (0, 0), (pad_eff,) * 2, (pad_eff,) * 2, (pad_eff,) * 2))
    Do, Ho, Wo = (v + 2 * pad_eff - k + 1 for v in (D, H, W))
    out = np.zeros((N, w.shape[1], Do, Ho, Wo))
    for a in range(k):
        for b in range(k):
            for c in range(k):
                patch = xp[:, :, a:a + Do, b:b + Ho, c:c + Wo]
                out += np.einsum("nidhw,oi->nodhw", patch, wf[:, :, a, b, c])
    return out


@pytest.mark.parametrize("k,p", [(2, 0), (3, 0), (3, 1), (4, 2), (5, 0), (5, 3)])
def test_stride1_equals_flipped_correlation(k, p):
    rng = np.random.default_rng(100 + 10 * k + p)
    x, w, _ = rand_case(rng, 2, 3, 4, 5, 6, 7, k, bias=False)
    Y = oracle.convt3d_scatter(x, w, None, stride=1, pad=p)
    ref = _flipped_correlation(x, w, k - 1 - p)
    assert Y.shape == ref.shape
    assert np.max(np.abs(Y - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


# ---------------------------------------------------- adjoint identity ----

def _forward_conv(y, w, s, p, in_shape):
    """Independent strided forward correlation with the same weight:
    out[n,ci,i] = sum_{co,t} w[ci,co,t] * y[n,co,i*s - p + t] (in-range terms)."""
    N = y.shape[0]
    Cin, Cout, k = w.shape[0], w.shape[1], w.shape[2]
    D, H, W = in_shape
    Do, Ho, Wo = y.shape[2:]
    out = np.zeros((N, Cin, D, H, W))
    w64 = w.astype(np.float64)
    for td in range(k):
        od = np.arange(D) * s - p + td
        md = (od >= 0) & (od < Do)
        for th in range(k):
            oh = np.arange(H) * s - p + th
            mh = (oh >= 0) & (oh < Ho)
            for tw in range(k):
                ow = np.arange(W) * s - p + tw
                mw = (ow >= 0) & (ow < Wo)
                g = y[:, :, np.clip(od, 0, Do - 1)][:, :, :, np.clip(oh, 0, Ho - 1)][:, :, :, :, np.clip(ow, 0, Wo - 1)]
                mask = md[:, None, None] & mh[None, :, None] & mw[None, None, :]
                out += np.einsum("nodhw,io->nidhw", g * mask, w64[:, :, td, th, tw])
    return out


@pytest.mark.parametrize("k,s,p,op", [(3, 1, 0, 0), (3, 2, 1, 1), (4, 2, 1, 0), (3, 3, 1, 2),
                                      (5, 2, 2, 1), (2, 2, 0, 0), (4, 3, 0, 1)])
def test_adjoint_identity(k, s, p, op):
    rng = np.random.default_rng(7 + 100 * k + 10 * s + p + 1000 * op)
    x, w, _ = rand_case(rng, 2, 3, 4, 4, 5, 3, k, bias=False)
    Y = oracle.convt3d_scatter(x, w, None, stride=s, pad=p, out_pad=op)
    yr = rng.standard_normal(Y.shape)
    lhs = float(np.sum(Y * yr))
    rhs = float(np.sum(x.astype(np.float64) * _forward_conv(yr, w, s, p, x.shape[2:])))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_linearity_and_bias():
    rng = np.random.default_rng(5)
    _, w, b = rand_case(rng, 2, 3, 4, 3, 4, 5, 3)
    # inputs on a coarse dyadic grid so that a1*x1 + a2*x2 is exact in fp32
    x1 = (rng.integers(-64, 65, (2, 3, 3, 4, 5)) / 32.0).astype(np.float32)
    x2 = (rng.integers(-64, 65, (2, 3, 3, 4, 5)) / 32.0).astype(np.float32)
    a1, a2 = 0.75, -1.5
    xs = (a1 * x1 + a2 * x2).astype(np.float32)
    for s, p, op in [(1, 0, 0), (2, 1, 1)]:
        Y1 = oracle.convt3d_scatter(x1, w, None, stride=s, pad=p, out_pad=op)
        Y2 = oracle.convt3d_scatter(x2, w, None, stride=s, pad=p, out_pad=op)
        Ys = oracle.convt3d_scatter(xs, w, None, stride=s, pad=p, out_pad=op)
        ref = a1 * Y1 + a2 * Y2
        assert np.max(np.abs(Ys - ref)) <= 1e-12 * np.max(np.abs(ref))
        Yb = oracle.convt3d_scatter(x1, w, b, stride=s, pad=p, out_pad=op)
        assert np.allclose(Yb - Y1, b.astype(np.float64)[None, :, None, None, None], atol=1e-15, rtol=0)


# --------------------------------------- library routine on special cases ----

@pytest.mark.parametrize("k,s,p,op", [(3, 1, 0, 0), (5, 1, 0, 0), (3, 2, 1, 1), (4, 2, 1, 0),
                                      (3, 1, 1, 0), (2, 3, 0, 2)])
def test_scatter_matches_torch_cpu_fp64(k, s, p, op):
    rng = np.random.default_rng(11 * k + s + 3 * p + 7 * op)
    x, w, b = rand_case(rng, 2, 5, 6, 4, 3, 5, k)
    Y = oracle.convt3d_scatter(x, w, b, stride=s, pad=p, out_pad=op)
    ref = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                             torch.from_numpy(b).double(), stride=s, padding=p,
                             output_padding=op).numpy()
    assert Y.shape == ref.shape
    assert np.max(np.abs(Y - ref)) <= 1e-12


# ------------------------------------------------- pooled-sum closed form ----

@pytest.mark.parametrize("k", [3, 5])
def test_pooled_sum_closed_form(k):
    # l2_p77: with stride 1 and no padding every tap of every input lands inside,
    # so sum_spatial Y[n,c] = sum_ci Xsum[n,ci] * Wsum[ci,c] + V * b[c].
    rng = np.random.default_rng(31 + k)
    x, w, b = rand_case(rng, 3, 4, 5, 4, 6, 5, k)
    Y = oracle.convt3d_scatter(x, w, b, stride=1, pad=0)
    V = np.prod(Y.shape[2:])
    xsum = x.astype(np.float64).sum(axis=(2, 3, 4))
    wsum = w.astype(np.float64).sum(axis=(2, 3, 4))
    closed = xsum @ wsum + V * b.astype(np.float64)[None, :]
    got = Y.sum(axis=(2, 3, 4))
    assert np.max(np.abs(got - closed)) <= 1e-10 * max(1.0, np.max(np.abs(closed)))


# ------------------------------------------------------ epilogue pins ----

def test_groupnorm_invariants():
    rng = np.random.default_rng(41)
    x, w, b = rand_case(rng, 2, 4, 8, 4, 5, 6, 3)
    G, eps = 4, 1e-5
    Y = oracle.convt3d_scatter(x, w, b, stride=1, pad=0)
    v = np.maximum(Y, 0.0).reshape(2, G, -1)
    sig2 = v.var(axis=2)
    _, y64 = oracle.forward(x, w, b, epilogue=oracle.EPI_RELU_GROUPNORM, groups=G, eps=eps,
                            want_f64=True)
    g = y64.reshape(2, G, -1)
    assert np.max(np.abs(g.mean(axis=2))) < 1e-12
    assert np.max(np.abs(g.var(axis=2) - sig2 / (sig2 + eps))) < 1e-12
    # affine: gamma/beta act per channel on the normalised values
    gamma = rng.uniform(0.5, 1.5, 8).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, 8).astype(np.float32)
    _, ya = oracle.forward(x, w, b, epilogue=oracle.EPI_RELU_GROUPNORM, groups=G, eps=eps,
                           gamma=gamma, beta=beta, want_f64=True)
    back = (ya - beta.astype(np.float64)[None, :, None, None, None]) / gamma.astype(np.float64)[None, :, None, None, None]
    assert np.max(np.abs(back - y64)) < 1e-12


def test_groupnorm_matches_torch_cpu_fp64():
    rng = np.random.default_rng(43)
    x, w, _ = rand_case(rng, 2, 4, 8, 3, 4, 5, 3, bias=False)
    gamma = rng.uniform(0.5, 1.5, 8).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, 8).astype(np.float32)
    _, y64 = oracle.forward(x, w, None, epilogue=oracle.EPI_RELU_GROUPNORM, groups=2, eps=1e-5,
                            gamma=gamma, beta=beta, want_f64=True)
    t = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double())
    ref = F.group_norm(F.relu(t), 2, torch.from_numpy(gamma).double(),
                       torch.from_numpy(beta).double(), eps=1e-5).numpy()
    assert np.max(np.abs(y64 - ref)) < 1e-10


def test_softmax_sigmoid_invariants():
    rng = np.random.default_rng(47)
    x, w, b = rand_case(rng, 2, 3, 6, 3, 4, 5, 3)
    _, y64 = oracle.forward(x, w, b, stride=2, pad=1, out_pad=1,
                            epilogue=oracle.EPI_SOFTMAX_SIGMOID, want_f64=True)
    # sigmoid(t) = y  <=>  t = log(y / (1 - y)); the softmax weights t sum to 1
    t = np.log(y64 / (1.0 - y64))
    assert np.max(np.abs(t.sum(axis=1) - 1.0)) < 1e-12
    g = GOLDEN["softmax_sigmoid_range"]
    assert y64.min() > g["low_exclusive"]
    assert y64.max() <= 1.0 / (1.0 + math.exp(-1.0))
    assert abs(1.0 / (1.0 + math.exp(-1.0)) - g["high_inclusive_approx"]) < 1e-3
    # monotone in the conv output along channels
    Y = oracle.convt3d_scatter(x, w, b, stride=2, pad=1, out_pad=1)
    assert np.array_equal(np.argsort(Y, axis=1, kind="stable"), np.argsort(t, axis=1, kind="stable"))


def test_softmax_sigmoid_matches_torch_cpu_fp64():
    rng = np.random.default_rng(53)
    x, w, b = rand_case(rng, 2, 3, 6, 3, 4, 5, 3)
    _, y64 = oracle.forward(x, w, b, stride=2, pad=1, out_pad=1,
                            epilogue=oracle.EPI_SOFTMAX_SIGMOID, want_f64=True)
    t = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                           torch.from_numpy(b).double(), stride=2, padding=1, output_padding=1)
    ref = torch.sigmoid(torch.softmax(t, dim=1)).numpy()
    assert np.max(np.abs(y64 - ref)) < 1e-14


def test_batchnorm_pool_channel_means_equal_beta_and_closed_form():
    rng = np.random.default_rng(59)
    N, C = 3, 6
    x, w, b = rand_case(rng, N, 4, C, 4, 5, 3, 3)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, C).astype(np.float32)
    s, eps = 2.0, 1e-5
    _, out = oracle.forward(x, w, b, epilogue=oracle.EPI_SCALE_BATCHNORM_AVGPOOL, scale=s,
                            eps=eps, gamma=gamma, beta=beta, want_f64=True)
    out = out.reshape(N, C)
    # mean over n of the pooled normalised values is exactly beta_c
    assert np.max(np.abs(out.mean(axis=0) - beta.astype(np.float64))) < 1e-12
    # l2_p77's algebra: pooled BN from per-(n,c) sums S and per-c sums of squares Q
    Y = oracle.convt3d_scatter(x, w, b, stride=1, pad=0)
    V = np.prod(Y.shape[2:])
    S = Y.sum(axis=(2, 3, 4))
    Q = (Y * Y).sum(axis=(2, 3, 4)).sum(axis=0)
    mu = s * S.sum(axis=0) / (N * V)
    var = s * s * Q / (N * V) - mu * mu
    closed = gamma * (s * S / V - mu) / np.sqrt(var + eps) + beta
    assert np.max(np.abs(out - closed)) < 1e-9


def test_batchnorm_pool_matches_torch_cpu_fp64():
    rng = np.random.default_rng(61)
    N, C = 2, 5
    x, w, b = rand_case(rng, N, 3, C, 3, 4, 3, 3)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, C).astype(np.float32)
    _, out = oracle.forward(x, w, b, epilogue=oracle.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0,
                            eps=1e-5, gamma=gamma, beta=beta, want_f64=True)
    t = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                           torch.from_numpy(b).double()) * 2.0
    z = F.batch_norm(t, None, None, torch.from_numpy(gamma).double(),
                     torch.from_numpy(beta).double(), training=True, eps=1e-5)
    ref = F.adaptive_avg_pool3d(z, 1).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_identity_rounds_once_to_fp32():
    rng = np.random.default_rng(67)
    x, w, b = rand_case(rng, 1, 3, 4, 3, 3, 3, 4)
    y, y64 = oracle.forward(x, w, b, stride=2, pad=1, want_f64=True)
    assert np.array_equal(y, y64.astype(np.float32))


def test_rejects_bad_arguments():
    x = np.zeros((1, 2, 3, 3, 3), np.float32)
    w = np.zeros((2, 6, 3, 3, 3), np.float32)
    with pytest.raises(ValueError):
        oracle.forward(x, w, epilogue=oracle.EPI_RELU_GROUPNORM, groups=4)  # 6 % 4 != 0
    with pytest.raises(ValueError):
        oracle.forward(x, w, epilogue=7)


def test_batchnorm_eval_pool_matches_torch_cpu_fp64():
    rng = np.random.default_rng(71)
    N, C = 2, 5
    x, w, b = rand_case(rng, N, 3, C, 3, 4, 3, 3)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, C).astype(np.float32)
    rm = rng.uniform(-0.2, 0.2, C).astype(np.float32)
    rv = rng.uniform(0.5, 2.0, C).astype(np.float32)
    _, out = oracle.forward(x, w, b, epilogue=oracle.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=2.0, eps=1e-5,
                            gamma=gamma, beta=beta, running_mean=rm, running_var=rv, want_f64=True)
    t = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                           torch.from_numpy(b).double()) * 2.0
    z = F.batch_norm(t, torch.from_numpy(rm).double(), torch.from_numpy(rv).double(),
                     torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(), training=False, eps=1e-5)
    ref = F.adaptive_avg_pool3d(z, 1).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_batchnorm_running_stats_match_torch_cpu_fp64():
    rng = np.random.default_rng(73)
    N, C, m = 3, 4, 0.1
    x, w, b = rand_case(rng, N, 3, C, 3, 3, 4, 3)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, C).astype(np.float32)
    rm = rng.uniform(-0.2, 0.2, C).astype(np.float32)
    rv = rng.uniform(0.5, 2.0, C).astype(np.float32)
    rm_t, rv_t = torch.from_numpy(rm.copy()).double(), torch.from_numpy(rv.copy()).double()
    oracle.forward(x, w, b, epilogue=oracle.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, eps=1e-5, gamma=gamma,
                   beta=beta, running_mean=rm, running_var=rv, momentum=m)
    t = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                           torch.from_numpy(b).double()) * 2.0
    F.batch_norm(t, rm_t, rv_t, torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(),
                 training=True, momentum=m, eps=1e-5)
    # stored in fp32 after an fp64 update
    assert np.max(np.abs(rm - rm_t.numpy())) < 1e-6
    assert np.max(np.abs(rv - rv_t.numpy())) < 1e-6


def test_batchnorm_eval_with_batch_statistics_equals_training_output():
    # evaluation-mode normalisation with the batch's own mean and biased variance
    # reproduces the batch-statistics epilogue
    rng = np.random.default_rng(79)
    N, C, s = 2, 3, 0.5
    x, w, b = rand_case(rng, N, 2, C, 3, 3, 3, 3)
    Y = oracle.convt3d_scatter(x, w, b)
    z = s * Y
    mean = z.mean(axis=(0, 2, 3, 4)).astype(np.float32)
    var = z.var(axis=(0, 2, 3, 4))
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, C).astype(np.float32)
    _, train = oracle.forward(x, w, b, epilogue=oracle.EPI_SCALE_BATCHNORM_AVGPOOL, scale=s, gamma=gamma,
                              beta=beta, want_f64=True)
    # the stored statistics are fp32: the bound covers their rounding
    _, ev = oracle.forward(x, w, b, epilogue=oracle.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=s, gamma=gamma,
                           beta=beta, running_mean=mean, running_var=var.astype(np.float32), want_f64=True)
    assert np.max(np.abs(ev - train)) < 1e-5


# ------------------------------ general shapes: per-dimension, dilation, groups ----

GENERAL_CASES = [
    # (kd, kh, kw), stride, pad, out_pad, dilation, conv_groups
    ((3, 2, 4), (1, 2, 2), (1, 0, 2), (0, 1, 1), (1, 1, 1), 1),
    ((3, 3, 3), (1, 1, 1), (0, 1, 2), (0, 0, 0), (2, 1, 3), 1),
    ((2, 3, 3), (2, 1, 2), (0, 1, 1), (1, 0, 0), (1, 2, 2), 1),
    ((3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), 2),
    ((1, 3, 2), (1, 2, 1), (0, 1, 0), (0, 1, 0), (1, 1, 1), 4),
    ((3, 2, 3), (2, 2, 1), (2, 1, 1), (0, 1, 0), (3, 2, 1), 2),
]


def _general_case(rng, N, Cin, Cout, D, H, W, kk, G, bias=True):
    x = rng.standard_normal((N, Cin, D, H, W)).astype(np.float32)
    kv = kk[0] * kk[1] * kk[2]
    w = (rng.uniform(-1, 1, (Cin, Cout // G) + tuple(kk)) / math.sqrt(Cout * kv)).astype(np.float32)
    b = rng.uniform(-0.3, 0.3, Cout).astype(np.float32) if bias else None
    return x, w, b


@pytest.mark.parametrize("kk,s,p,op,dil,G", GENERAL_CASES)
def test_general_scatter_matches_torch_cpu_fp64(kk, s, p, op, dil, G):
    rng = np.random.default_rng(sum(kk) * 7 + sum(s) + 3 * sum(p) + 11 * sum(dil) + G)
    x, w, b = _general_case(rng, 2, 4, 8, 3, 4, 5, kk, G)
    Y = oracle.convt3d_scatter_general(x, w, b, stride=s, pad=p, out_pad=op, dilation=dil, conv_groups=G)
    ref = F.conv_transpose3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                             torch.from_numpy(b).double(), stride=s, padding=p, output_padding=op,
                             groups=G, dilation=dil).numpy()
    assert Y.shape == ref.shape
    assert np.max(np.abs(Y - ref)) <= 1e-12


def _forward_conv_general(y, w, s, p, dil, G, in_shape):
    """Independent strided, dilated, grouped forward correlation with the same weight:
    out[n,ci,i] = sum_{co in group(ci), t} w[ci,co',t] * y[n,co,i*s - p + dil*t]."""
    N = y.shape[0]
    Cin, Cout_g = w.shape[0], w.shape[1]
    Cin_g = Cin // G
    kd, kh, kw = w.shape[2:]
    out = np.zeros((N, Cin) + tuple(in_shape))
    Y = y
    Do, Ho, Wo = Y.shape[2:]
    w64 = w.astype(np.float64)
    for ci in range(Cin):
        g = ci // Cin_g
        for col in range(Cout_g):
            co = g * Cout_g + col
            for a in range(kd):
                for bb in range(kh):
                    for c in range(kw):
                        od = np.arange(in_shape[0]) * s[0] - p[0] + dil[0] * a
                        oh = np.arange(in_shape[1]) * s[1] - p[1] + dil[1] * bb
                        ow = np.arange(in_shape[2]) * s[2] - p[2] + dil[2] * c
                        md, mh, mw = (od >= 0) & (od < Do), (oh >= 0) & (oh < Ho), (ow >= 0) & (ow < Wo)
                        sub = Y[:, co][:, np.clip(od, 0, Do - 1)][:, :, np.clip(oh, 0, Ho - 1)][:, :, :, np.clip(ow, 0, Wo - 1)]
                        mask = md[:, None, None] & mh[None, :, None] & mw[None, None, :]
                        out[:, ci] += w64[ci, col, a, bb, c] * sub * mask
    return out


@pytest.mark.parametrize("kk,s,p,op,dil,G", GENERAL_CASES)
def test_general_adjoint_identity(kk, s, p, op, dil, G):
    rng = np.random.default_rng(1000 + sum(kk) + 5 * sum(dil) + G)
    x, w, _ = _general_case(rng, 1, 4, 4, 3, 3, 4, kk, G, bias=False)
    Y = oracle.convt3d_scatter_general(x, w, None, stride=s, pad=p, out_pad=op, dilation=dil, conv_groups=G)
    yr = rng.standard_normal(Y.shape)
    lhs = float(np.sum(Y * yr))
    rhs = float(np.sum(x.astype(np.float64) * _forward_conv_general(yr, w, s, p, dil, G, x.shape[2:])))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_groups_are_independent_dense_convolutions():
    # a grouped transposed convolution is G dense ones on channel slices, concatenated
    rng = np.random.default_rng(77)
    G, kk = 3, (3, 2, 3)
    x, w, b = _general_case(rng, 2, 6, 9, 3, 4, 3, kk, G)
    Y = oracle.convt3d_scatter_general(x, w, b, stride=(2, 1, 2), pad=(1, 0, 1), out_pad=(1, 0, 0), conv_groups=G)
    for g in range(G):
        xs = np.ascontiguousarray(x[:, 2 * g:2 * g + 2])
        ws = np.ascontiguousarray(w[2 * g:2 * g + 2])
        Yg = oracle.convt3d_scatter_general(xs, ws, np.ascontiguousarray(b[3 * g:3 * g + 3]), stride=(2, 1, 2),
                                            pad=(1, 0, 1), out_pad=(1, 0, 0))
        assert np.array_equal(Y[:, 3 * g:3 * g + 3], Yg)


def test_general_forward_epilogues_match_cubic_entry():
    # the general entry with cubic, dense, undilated arguments is the cubic one
    rng = np.random.default_rng(91)
    x, w, b = rand_case(rng, 2, 3, 8, 3, 4, 3, 3)
    gamma = rng.uniform(0.5, 1.5, 8).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, 8).astype(np.float32)
    a = oracle.forward(x, w, b, stride=2, pad=1, out_pad=1, epilogue=oracle.EPI_RELU_GROUPNORM, groups=2,
                       gamma=gamma, beta=beta)
    c = oracle.forward(x, w, b, stride=(2, 2, 2), pad=(1, 1, 1), out_pad=(1, 1, 1), dilation=(1, 1, 1),
                       conv_groups=1, epilogue=oracle.EPI_RELU_GROUPNORM, groups=2, gamma=gamma, beta=beta)
    assert np.array_equal(a, c)
