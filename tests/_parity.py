"""Comparison helpers shared by the GPU parity tests (test code only)."""

import numpy as np
import torch

from oracle import moe_oracle as o

# Floating-point contract: max |err| <= REL_RMS * RMS(ref) and cosine >= MIN_COS.
REL_RMS = 2e-2
MIN_COS = 0.9999


def with_gate_logits(t):
    """Layers whose logits are the gate projection of x come from the generator with
    W_g and logits None; the oracle projects them here and both sides get the same
    logits."""
    if t.get("logits") is None:
        lg = o.router_logits(bits_np(t["x"]), t["wg"].cpu().numpy()).astype(np.float32)
        t["logits"] = torch.from_numpy(lg).to(t["x"].device)
    return t


def bf16_np(t):
    """bf16 torch tensor (any device) -> float64 numpy."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits_np(t):
    """bf16 torch tensor -> uint16 bit patterns (numpy)."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_float_close(got, ref, name, rel=REL_RMS, min_cos=MIN_COS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    if rms == 0.0:
        assert err == 0.0, f"{name}: reference is zero, max err {err}"
        return dict(max_err=err, rms=0.0, cos=1.0)
    cos = float(np.dot(got.ravel(), ref.ravel()) /
                (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-300))
    assert err <= rel * rms, f"{name}: max|err| {err:.4g} > {rel} * RMS {rms:.4g}"
    assert cos >= min_cos, f"{name}: cosine {cos:.7f} < {min_cos}"
    return dict(max_err=err, rms=rms, cos=cos)


def fp8_rows_dequant(q, s):
    return o.dequant_rows(np.asarray(q), np.asarray(s))


def assert_fp8_codes_close(gq, gs, rq, rs, name, max_mismatch=1e-2):
    """FP8 codes produced from floating-point inputs on both sides: scales and codes
    must agree except for rare ties broken differently by last-bit differences
    upstream; every differing code must be the neighbouring value after scaling.
    Returns the code agreement rate."""
    gq, gs, rq, rs = (np.asarray(a) for a in (gq, gs, rq, rs))
    assert gq.shape == rq.shape and gs.shape == rs.shape
    sc_mis = np.mean(gs != rs) if gs.size else 0.0
    assert sc_mis <= max_mismatch, f"{name}: scale mismatch rate {sc_mis}"
    gd = fp8_rows_dequant(gq, gs)
    rd = fp8_rows_dequant(rq, rs)
    mis = gq != rq
    rate = float(np.mean(mis)) if mis.size else 0.0
    assert rate <= max_mismatch, f"{name}: code mismatch rate {rate}"
    if mis.any():
        # a differing code is at most one E4M3 step (relative 2^-3, or one subnormal
        # step) away from the reference after dequantisation
        scale = o.e8m0_decode(np.repeat(rs, 128, axis=1))
        step = np.maximum(np.abs(rd) * 2.0 ** -3, scale * 2.0 ** -9) * 1.0001
        # where the block scales differ the values may move by one binade step
        step = np.where(np.repeat(gs != rs, 128, axis=1), np.abs(rd) + scale, step)
        assert np.all(np.abs(gd - rd)[mis] <= step[mis]), f"{name}: non-adjacent code"
    return 1.0 - rate
