"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method: it only draws random numbers
(torch's CPU generator, fixed seeds) and rounds them to BF16 with torch's own
cast.  Both the CUDA library's callers and the CPU oracle's callers take their
inputs from here, so the two sides see the same bits.

The five workloads mirror the shapes of the paper's MoE rollout and QAT
settings (QUADS §4.1) at kernel level:

  1 dense_small   X 64x512 ~N(0,1), 4 outlier channels x50; W 512x512 ~N(0,.02); k=16
  2 dense_decode  X 256x4096 Student-t(4), 32 outlier channels x30;
                  W 4096x4096 ~N(0,.02); k=128
  3 moe_decode    2048 tokens, hidden 2048, 64 experts top-8 (softmax of N(0,1)
                  logits), gate_up 2048->2x768, down 768->2048, SwiGLU, k=64
  4 qat           fake-quant of 128 experts x {gate_up 3072x4096, down 4096x1536},
                  then the BF16-activation GEMM on 4096 tokens routed top-8
  5 moe_prefill   16384 tokens, hidden 4096, 128 experts top-8 with Zipf(1.1)
                  routing, intermediate 1536, SwiGLU, X Student-t(3) with 64
                  outlier channels x50, k=128
"""
import torch

CONFIGS = {
    1: dict(name="dense_small", kind="dense", M=64, K=512, N=512, k=16,
            law="normal", n_outliers=4, outlier_scale=50.0),
    2: dict(name="dense_decode", kind="dense", M=256, K=4096, N=4096, k=128,
            law="student_t", nu=4, n_outliers=32, outlier_scale=30.0),
    3: dict(name="moe_decode", kind="moe", T=2048, H=2048, E=64, topk=8, I=768, k=64,
            law="normal", n_outliers=0, outlier_scale=1.0, routing="normal"),
    4: dict(name="qat", kind="qat", T=4096, H=4096, E=128, topk=8, I=1536, k=0,
            law="normal", n_outliers=0, outlier_scale=1.0, routing="normal"),
    5: dict(name="moe_prefill", kind="moe", T=16384, H=4096, E=128, topk=8, I=1536, k=128,
            law="student_t", nu=3, n_outliers=64, outlier_scale=50.0, routing="zipf"),
}

# sub-stream ids of the seeds
_X, _W, _LOGITS, _OUTLIERS, _PERM, _W13, _DOWN = 1, 2, 3, 4, 5, 100, 200


def _gen(cfg_id, stream, sub=0):
    g = torch.Generator(device="cpu")
    g.manual_seed(((1000 + cfg_id) * 1000 + stream) * 100003 + sub)
    return g


def _draw(law, shape, g, nu=None):
    if law == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float64)
    if law == "student_t":
        z = torch.randn(shape, generator=g, dtype=torch.float64)
        chi2 = torch.zeros(shape, dtype=torch.float64)
        for _ in range(nu):
            chi2 += torch.randn(shape, generator=g, dtype=torch.float64) ** 2
        return z / torch.sqrt(chi2 / nu)
    raise ValueError(law)


def outlier_channels(cfg_id):
    """Seeded positions of the outlier channels (sorted), shared by every batch."""
    c = CONFIGS[cfg_id]
    K = c.get("K", c.get("H"))
    if c["n_outliers"] == 0:
        return torch.zeros(0, dtype=torch.int64)
    perm = torch.randperm(K, generator=_gen(cfg_id, _OUTLIERS))
    return torch.sort(perm[: c["n_outliers"]]).values


def activations(cfg_id, batch=0, rows=None):
    """BF16 activations [M, K] of a workload.  batch=1 is the calibration batch
    (an independent draw with the same outlier channel positions)."""
    c = CONFIGS[cfg_id]
    M = c.get("M", c.get("T")) if rows is None else rows
    K = c.get("K", c.get("H"))
    x = _draw(c["law"], (M, K), _gen(cfg_id, _X, batch), c.get("nu"))
    oc = outlier_channels(cfg_id)
    if oc.numel():
        x[:, oc] *= c["outlier_scale"]
    return x.to(torch.bfloat16)


def dense_weight(cfg_id):
    """BF16 weight [N, K] ~ N(0, 0.02) of a dense workload."""
    c = CONFIGS[cfg_id]
    w = torch.randn((c["N"], c["K"]), generator=_gen(cfg_id, _W), dtype=torch.float32) * 0.02
    return w.to(torch.bfloat16)


def expert_weight(cfg_id, e, proj):
    """BF16 weight of expert e: proj 'w13' -> [2I, H] (gate rows then up rows),
    'down' -> [H, I].  Each expert has its own seed, so any one expert can be
    regenerated alone."""
    c = CONFIGS[cfg_id]
    shape = (2 * c["I"], c["H"]) if proj == "w13" else (c["H"], c["I"])
    stream = _W13 if proj == "w13" else _DOWN
    w = torch.randn(shape, generator=_gen(cfg_id, stream, e), dtype=torch.float32) * 0.02
    return w.to(torch.bfloat16)


def router_logits(cfg_id):
    """Router logits float32 [T, E].  'normal': N(0,1).  'zipf': Gumbel(0,1)
    noise plus log p_e with p_e proportional to (rank_e + 1)^-1.1 over a seeded
    permutation of the experts, so that top-k of the logits samples k distinct
    experts without replacement with Zipf(1.1) popularity."""
    c = CONFIGS[cfg_id]
    T, E = c["T"], c["E"]
    g = _gen(cfg_id, _LOGITS)
    if c["routing"] == "normal":
        return torch.randn((T, E), generator=g, dtype=torch.float32)
    rank = torch.randperm(E, generator=_gen(cfg_id, _PERM)).to(torch.float64)
    logp = -1.1 * torch.log(rank + 1.0)
    logp = logp - torch.logsumexp(logp, 0)
    u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_min(1e-300)
    gumbel = -torch.log(-torch.log(u))
    return (gumbel + logp[None, :]).to(torch.float32)


def engine_drift(x, rel, seed):
    """Synthetic engine drift eta (QUADS §3.1 Eq. 8): the inference engine's
    copy of a BF16 activation x, bf16(x * (1 + rel * z)) with z ~ N(0, 1)
    seeded per element -- a relative perturbation of about rel, standing in
    for the different reduction orders of two engines."""
    g = torch.Generator(device="cpu")
    g.manual_seed(7919 * 100003 + seed)
    z = torch.randn(x.shape, generator=g, dtype=torch.float64)
    return (x.double() * (1.0 + rel * z)).to(torch.bfloat16)


def u16(t):
    """BF16 torch tensor -> numpy uint16 bit patterns (for the oracle)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def flops_moe(cfg_id):
    """(fp4 flops, bf16 RAC flops) of one MoE layer forward of a workload."""
    c = CONFIGS[cfg_id]
    R = c["T"] * c["topk"]
    f4 = 2 * R * (2 * c["I"]) * c["H"] + 2 * R * c["H"] * c["I"]
    fb = 2 * R * (2 * c["I"]) * c["k"] + 2 * R * c["H"] * c["k"]
    return f4, fb


def describe(cfg_id):
    c = CONFIGS[cfg_id]
    return {k: v for k, v in c.items()}

