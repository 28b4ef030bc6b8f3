"""Seeded synthetic inputs for the routed MoE expert FFN.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no quantisation, routing, GEMM or activation).  The CUDA path
and the oracle both receive exactly these tensors.

Workloads (shapes from the MoE layers described in "Pushing the Limits of Serving
DeepSeek-V4-Pro" -- 384 routed experts, one shared expert -- and the GB10
"Optimization progress report" -- 7-token verify steps):

  tiny    T=64    H=512  I=256  E=8   k=2  no shared expert
  decode  T=7     H=7168 I=3072 E=384 k=8  + shared expert, logits ~ N(0, 1)
  decode256  T=256  same dims, Zipf(1.1) expert popularity
  prefill  T=32768 same dims, Zipf(1.1) expert popularity
  sweep   grouped-GEMM sweep, W13 (N=6144, K=7168) and W2 (N=7168, K=3072)

Weights are MXFP4: E2M1 code bytes uniform over all 256 values (so each nibble is
uniform over the 16 codes), E8M0 scale bytes uniform over {123..127} (exponent
uniform in [-4, 0]).  The NVFP4 form (nvfp4_layer_weights) draws the same code
bytes, E4M3 block scales uniform over the 40 positive codes 2^-4 .. 1.875, and fp32
tensor scales uniform in [0.5, 1.5).  Activations are bf16 N(0, 1).

Router logits:
  tiny:            logits = the gate projection x . W_g^T with W_g fp32 ~ N(0, 0.02);
      this module draws W_g only, the projection is a step of the method (the
      oracle computes it in the tests, the library's router kernel in the benchmark);
  decode:          logits fp32 ~ N(0, 1);
  decode256/prefill: logits = fp32(bias_e + g), g standard Gumbel noise and
      bias_e = -1.1 * ln(rank(e)), rank from a seeded permutation of the experts;
      Gumbel-top-k then draws experts without replacement with probability
      proportional to rank**-1.1 (Zipf, s = 1.1).
"""

from __future__ import annotations

import dataclasses
import torch


@dataclasses.dataclass(frozen=True)
class Dims:
    T: int
    H: int
    I: int
    E: int
    k: int
    has_shared: int

    @property
    def G(self) -> int:
        return self.E + self.has_shared

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def Rs(self) -> int:
        return self.R + (self.T if self.has_shared else 0)


WORKLOADS = {
    "tiny": Dims(T=64, H=512, I=256, E=8, k=2, has_shared=0),
    "decode": Dims(T=7, H=7168, I=3072, E=384, k=8, has_shared=1),
    "decode256": Dims(T=256, H=7168, I=3072, E=384, k=8, has_shared=1),
    "prefill": Dims(T=32768, H=7168, I=3072, E=384, k=8, has_shared=1),
}
LOGITS_KIND = {"tiny": "gate", "decode": "normal", "decode256": "zipf", "prefill": "zipf"}

SWEEP_M = (1, 2, 4, 7, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)
SWEEP_SHAPES = {"w13": (6144, 7168), "w2": (7168, 3072)}  # (N, K)


def sweep_groups(M: int) -> int:
    """Number of groups at per-group M in the GEMM sweep: G*M ~ 32768 for M >= 64,
    G = 64 below."""
    return 32768 // M if M >= 64 else 64


# Fixed order of the per-tensor seeds.
_STREAMS = ("x", "gate", "logits", "perm", "w13", "w13_s", "w2", "w2_s", "act")


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _STREAMS.index(name))
    return g


def mxfp4_weights(G, N, K, seed, device, name="w13", exp_lo=-4, exp_hi=0):
    """Random MXFP4 matrices: code bytes u8 [G, N, K/2], E8M0 bytes u8 [G, N, K/32]."""
    codes = torch.randint(0, 256, (G, N, K // 2), generator=_gen(seed, name, device),
                          device=device, dtype=torch.uint8)
    scales = torch.randint(127 + exp_lo, 127 + exp_hi + 1, (G, N, K // 32),
                           generator=_gen(seed, name + "_s", device), device=device,
                           dtype=torch.uint8)
    return codes, scales


# NVFP4 block scales: positive E4M3 codes with exponent field 3..7 and any mantissa,
# i.e. values 2^-4 .. 1.875 (the same binades as the MXFP4 scales above).
NVFP4_SCALE_CODES = tuple((e << 3) | m for e in range(3, 8) for m in range(8))


def nvfp4_weights(G, N, K, seed, device, name="w13", segments=1):
    """Random NVFP4 matrices: code bytes u8 [G, N, K/2] (each nibble uniform over the
    16 E2M1 codes), E4M3 block-scale bytes u8 [G, N, K/16] uniform over
    NVFP4_SCALE_CODES, fp32 tensor scales [G, segments] uniform in [0.5, 1.5)."""
    codes = torch.randint(0, 256, (G, N, K // 2), generator=_gen(seed, name, device),
                          device=device, dtype=torch.uint8)
    table = torch.tensor(NVFP4_SCALE_CODES, dtype=torch.uint8, device=device)
    i = torch.randint(0, len(table), (G, N, K // 16), generator=_gen(seed, name + "_s", device),
                      device=device)
    gs = 0.5 + torch.rand(G, segments, generator=_gen(seed, name + "_s", "cpu"),
                          dtype=torch.float32)
    return codes, table[i], gs.to(device)


def nvfp4_layer_weights(d, seed=0, device="cpu"):
    """NVFP4 expert weights of a layer: w13 [G, 2I, H/2] + w13_s [G, 2I, H/16] + w13_gs
    [G, 2] (gate rows, up rows), w2 [G, H, I/2] + w2_s [G, H, I/16] + w2_gs [G]."""
    w13, w13_s, w13_gs = nvfp4_weights(d.G, 2 * d.I, d.H, seed, device, "w13", segments=2)
    w2, w2_s, w2_gs = nvfp4_weights(d.G, d.H, d.I, seed, device, "w2", segments=1)
    return dict(w13=w13, w13_s=w13_s, w13_gs=w13_gs, w2=w2, w2_s=w2_s,
                w2_gs=w2_gs.reshape(d.G))


def activations(T, H, seed, device, name="x"):
    return torch.randn(T, H, generator=_gen(seed, name, device), device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def zipf_logits(T, E, seed, device, s=1.1):
    perm = torch.randperm(E, generator=_gen(seed, "perm", "cpu"), device="cpu")
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    bias = (-s * torch.log(rank)).to(device)
    u = torch.rand(T, E, generator=_gen(seed, "logits", device), device=device,
                   dtype=torch.float64)
    u = u.clamp_(min=1e-300)
    gumbel = -torch.log(-torch.log(u))
    return (bias[None, :] + gumbel).to(torch.float32)


def gate_weight(E, H, seed, device):
    """Router gate weight W_g fp32 [E, H], N(0, 0.02^2) entries."""
    return (torch.randn(E, H, generator=_gen(seed, "gate", "cpu"), dtype=torch.float32)
            * 0.02).to(device)


def router_logits(kind, x, E, seed, device):
    """Router logits drawn directly ("normal", "zipf"); for "gate" the logits are the
    gate projection of x, which is a step of the method, not of input generation: the
    layer then carries W_g (`gate_weight`) and logits None, and the caller projects
    (the oracle in the tests, the library's router kernel in the benchmark)."""
    T, H = x.shape
    if kind == "gate":
        return None
    if kind == "normal":
        return torch.randn(T, E, generator=_gen(seed, "logits", device), device=device,
                           dtype=torch.float32)
    if kind == "zipf":
        return zipf_logits(T, E, seed, device)
    raise ValueError(kind)


def make_layer(workload: str, seed: int = 0, device="cpu", T: int | None = None):
    """All inputs of one MoE layer: x bf16 [T, H], logits fp32 [T, E] and MXFP4
    W13 [G, 2I, H/2] + [G, 2I, H/32], W2 [G, H, I/2] + [G, H, I/32].
    `T` overrides the token count (same per-token recipe)."""
    d = WORKLOADS[workload]
    if T is not None:
        d = dataclasses.replace(d, T=T)
    x = activations(d.T, d.H, seed, device)
    logits = router_logits(LOGITS_KIND[workload], x, d.E, seed, device)
    wg = gate_weight(d.E, d.H, seed, device) if logits is None else None
    w13, w13_s = mxfp4_weights(d.G, 2 * d.I, d.H, seed, device, "w13")
    w2, w2_s = mxfp4_weights(d.G, d.H, d.I, seed, device, "w2")
    return d, dict(x=x, logits=logits, wg=wg, w13=w13, w13_s=w13_s, w2=w2, w2_s=w2_s)


def custom_layer(d: Dims, seed: int = 0, device="cpu", logits_kind="normal"):
    """Same recipe at arbitrary dims (ragged / edge-case tests)."""
    x = activations(d.T, d.H, seed, device)
    logits = router_logits(logits_kind, x, d.E, seed, device)
    wg = gate_weight(d.E, d.H, seed, device) if logits is None else None
    w13, w13_s = mxfp4_weights(d.G, 2 * d.I, d.H, seed, device, "w13")
    w2, w2_s = mxfp4_weights(d.G, d.H, d.I, seed, device, "w2")
    return dict(x=x, logits=logits, wg=wg, w13=w13, w13_s=w13_s, w2=w2, w2_s=w2_s)


def sweep_point(which: str, M: int, seed: int = 0, device="cpu", G: int | None = None):
    """One point of the grouped-GEMM sweep: G groups of M rows each.  Returns
    (x bf16 [G*M, K] activations to be quantised, group offsets int32 [G+1],
    W codes, W scales)."""
    N, K = SWEEP_SHAPES[which]
    G = sweep_groups(M) if G is None else G
    x = activations(G * M, K, seed, device, name="act")
    offsets = torch.arange(0, G + 1, dtype=torch.int32) * M
    w, ws = mxfp4_weights(G, N, K, seed, device, "w13" if which == "w13" else "w2")
    return x, offsets.to(device), w, ws


# --- exact-integer inputs: every product exact, partial sums < 2**24 -----------------

# E4M3 code bytes of the integers 0, +-1 .. +-8 (0x38 = 1.0, 0x40 = 2.0, ... 0x50 = 8.0;
# bit 7 is the sign).  -0 (0x80) is left out.
E4M3_INTEGER_CODES = (0x00, 0x38, 0xB8, 0x40, 0xC0, 0x44, 0xC4, 0x48, 0xC8,
                      0x4A, 0xCA, 0x4C, 0xCC, 0x4E, 0xCE, 0x50, 0xD0)
# E2M1 codes with integer values {0, +-1, +-2, +-3, +-4, +-6}.
E2M1_INTEGER_CODES = (0x0, 0x2, 0x4, 0x5, 0x6, 0x7, 0xA, 0xC, 0xD, 0xE, 0xF)


def integer_codes(shape, table, seed, device, name):
    t = torch.tensor(table, dtype=torch.uint8, device=device)
    i = torch.randint(0, len(table), shape, generator=_gen(seed, name, device), device=device)
    return t[i]


def integer_fp4_bytes(shape, seed, device, name):
    lo = integer_codes(shape, E2M1_INTEGER_CODES, seed, device, name)
    hi = integer_codes(shape, E2M1_INTEGER_CODES, seed + 7919, device, name)
    return lo | (hi << 4)
