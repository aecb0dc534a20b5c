"""Pins for the oracle's composed forward.

The composed forward (route -> gather -> GEMM -> silu_mul -> GEMM -> combine)
is checked against the dense masked formulation of BaselineMoE._forward in
mslk/moe/layers.py, written here in float64 numpy: every expert runs on every
token with the router score scattered into an [E, T] mask, and the expert
outputs are summed.  The two formulations share no code; a dropped score, a
swapped SwiGLU half, a transposed weight or a wrong combine breaks the match.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_token_routing_index_gb300 import workloads
from tests.helpers import bits, f64, rms


def dense_forward(x, scores, w13, w2, top_k, Tv):
    """BaselineMoE._forward restricted to the routed experts, float64, no rounding."""
    T, D = x.shape
    E = scores.shape[1]
    H = w2.shape[2]
    s = scores[:Tv]
    top = np.argsort(-s, axis=1, kind="stable")[:, :top_k]      # torch.topk, lower index on ties
    masked = np.zeros_like(s)
    np.put_along_axis(masked, top, np.take_along_axis(s, top, 1), 1)
    out = np.zeros((Tv, D))
    for e in range(E):
        xt = x[:Tv] * masked[:, e:e + 1]                          # tokens * masked_scores
        y = xt @ w13[e].T
        y0, y1 = y[:, :H], y[:, H:]
        z = y0 * (1 / (1 + np.exp(-y0))) * y1
        out += z @ w2[e].T
    return out


def _close(got, ref, rel_l2, max_rms):
    """Relative L2 error and max error against the unrounded dense reference.

    The composed forward rounds to bf16 (or e4m3) at every stage boundary and
    the dense reference rounds nowhere, so they differ by the accumulated
    rounding: about 0.3% of rms on average for bf16, with tails of a few percent.
    Mistakes in the composition give errors of order the signal itself.
    """
    err = got - ref
    l2 = np.linalg.norm(err) / np.linalg.norm(ref)
    mx = np.abs(err).max() / rms(ref)
    assert l2 <= rel_l2 and mx <= max_rms, (l2, mx)


def _problem(seed, T, D, H, E, k, std, Tv=None, fp8=False):
    cfg = workloads.MoEConfig("pin", T=T, D=D, H=H, E=E, top_k=k, Tv=Tv, fp8=fp8, weight_std=std)
    x = workloads.make_tokens(cfg, seed)
    s = workloads.make_scores(cfg, seed)
    w13, w2 = workloads.make_weights(cfg, seed)
    return cfg, x, s, w13, w2


@pytest.mark.parametrize("k,Tv", [(1, None), (2, None), (3, 37)])
def test_bf16_forward_matches_dense_formulation(k, Tv):
    cfg, x, s, w13, w2 = _problem(5, T=48, D=64, H=32, E=5, k=k, std=0.15, Tv=Tv)
    weights = lambda ids: (bits(w13[ids]), bits(w2[ids]))
    res = oracle.moe_forward(bits(x), bits(s), k, weights, fp8=False, valid_tokens=Tv)
    tv = cfg.valid_tokens
    ref = dense_forward(x.double().numpy(), s.double().numpy(), w13.double().numpy(),
                        w2.double().numpy(), k, tv)
    got = f64(res["out"])
    _close(got[:tv], ref, 1e-2, 0.1)
    assert np.all(res["out"][tv:] == 0), "tokens past the valid count stay as initialised"


def _fake_quant_rows(v):
    """Quantise rows to e4m3 with torch's own cast and dequantise (float64).

    Row rule of BaselineMoE._fake_quant's per-row quantiser: scale the row so
    that its largest magnitude is 448; an all-zero row stays zero.
    """
    m = np.abs(v).max(axis=-1, keepdims=True)
    s = np.where(m > 0, 448.0 / np.where(m > 0, m, 1), 1.0)
    q = torch.from_numpy((v * s).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    return q / s


def dense_forward_fake_quant(x, scores, w13, w2, top_k, z_bf16=False):
    """BaselineMoE._forward with _fake_quant on both GEMMs, float64 elsewhere
    (z_bf16: z rounded to bf16 before its quantisation, as routed_z is a bf16
    tensor there)."""
    T, D = x.shape
    E = scores.shape[1]
    H = w2.shape[2]
    top = np.argsort(-scores, axis=1, kind="stable")[:, :top_k]
    masked = np.zeros_like(scores)
    np.put_along_axis(masked, top, np.take_along_axis(scores, top, 1), 1)
    out = np.zeros((T, D))
    for e in range(E):
        xt = _fake_quant_rows(x * masked[:, e:e + 1])
        y = xt @ _fake_quant_rows(w13[e]).T
        y0, y1 = y[:, :H], y[:, H:]
        z = y0 * (1 / (1 + np.exp(-y0))) * y1
        if z_bf16:
            z = torch.from_numpy(z).to(torch.bfloat16).double().numpy()
        z = _fake_quant_rows(z)
        out += z @ _fake_quant_rows(w2[e]).T
    return out


@pytest.mark.parametrize("z_bf16", [False, True])
def test_fp8_forward_matches_dense_formulation(z_bf16):
    cfg, x, s, w13, w2 = _problem(6, T=40, D=64, H=48, E=4, k=2, std=0.15, fp8=True)
    weights = lambda ids: (w13[ids].numpy(), w2[ids].numpy())
    res = oracle.moe_forward(bits(x), bits(s), 2, weights, fp8=True, scale_ub=1200.0, z_bf16=z_bf16)
    got = f64(res["out"])
    args = (x.double().numpy(), s.double().numpy(), w13.double().numpy(), w2.double().numpy(), 2)
    # Against the unquantised math the four e4m3 roundings (3 mantissa bits
    # each) leave about 6% relative L2 error.
    _close(got, dense_forward(*args, cfg.T), 0.1, 0.6)
    # Against the same math with the fake-quantised GEMMs only the bf16
    # roundings between stages remain.
    _close(got, dense_forward_fake_quant(*args, z_bf16=z_bf16), 2e-2, 0.2)
    if z_bf16:   # the bf16 z is the one quantised: the composition's z stage equals silu_mul's output
        zq, zs = oracle.quantize_rows(oracle.bf16_to_f32(oracle.silu_mul(res["y"], 48)), 1200.0)
        np.testing.assert_array_equal(res["z"], zq)
        np.testing.assert_array_equal(res["z_scale"], zs)


def test_scaling_is_applied_to_the_expert_input():
    # f(s * x) differs from s * f(x) through the SiLU; the pages scale the input.
    cfg, x, s, w13, w2 = _problem(7, T=32, D=32, H=16, E=3, k=1, std=0.3)
    weights = lambda ids: (bits(w13[ids]), bits(w2[ids]))
    got = f64(oracle.moe_forward(bits(x), bits(s), 1, weights, fp8=False)["out"])
    sv = s.double().numpy()
    e = np.argsort(-sv, axis=1, kind="stable")[:, 0]
    sel = sv[np.arange(32), e][:, None]
    out_scaled = np.zeros((32, 32))
    for t in range(32):
        y = x[t].double().numpy() @ w13[e[t]].double().numpy().T
        z = y[:16] / (1 + np.exp(-y[:16])) * y[16:]
        out_scaled[t] = sel[t] * (z @ w2[e[t]].double().numpy().T)
    ref = dense_forward(x.double().numpy(), sv, w13.double().numpy(), w2.double().numpy(), 1, 32)
    _close(got, ref, 1e-2, 0.1)
    assert np.linalg.norm(got - out_scaled) > 0.1 * np.linalg.norm(ref)


def test_out_init_is_accumulated_into():
    cfg, x, s, w13, w2 = _problem(8, T=24, D=32, H=16, E=4, k=2, std=0.1)
    weights = lambda ids: (bits(w13[ids]), bits(w2[ids]))
    init = bits(torch.full((24, 32), 3.0, dtype=torch.bfloat16))
    a = oracle.moe_forward(bits(x), bits(s), 2, weights, fp8=False)
    b = oracle.moe_forward(bits(x), bits(s), 2, weights, fp8=False, out_init=init)
    np.testing.assert_allclose(f64(b["out"]), f64(a["out"]) + 3.0, atol=2 ** -6 * 4)


@pytest.mark.parametrize("fp8,z_bf16", [(False, False), (True, False), (True, True)])
def test_sampled_tokens_equal_the_full_forward(fp8, z_bf16):
    cfg, x, s, w13, w2 = _problem(9, T=30, D=32, H=16, E=6, k=2, std=0.1, fp8=fp8)
    if fp8:
        weights = lambda ids: (w13[ids].numpy(), w2[ids].numpy())
    else:
        weights = lambda ids: (bits(w13[ids]), bits(w2[ids]))
    full = oracle.moe_forward(bits(x), bits(s), 2, weights, fp8=fp8, scale_ub=1200.0, z_bf16=z_bf16)
    sample = np.array([0, 7, 8, 29])
    part, _ = oracle.moe_forward_tokens(sample, bits(x), bits(s), 2, weights, fp8=fp8, scale_ub=1200.0,
                                        z_bf16=z_bf16)
    np.testing.assert_array_equal(part, full["out"][sample])
