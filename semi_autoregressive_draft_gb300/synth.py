"""Seeded synthetic inputs for the draft/verify hot path.

This module only draws inputs; it contains none of the method's arithmetic.
Both the CUDA path's tests/benchmark and the CPU oracle read what it returns.

Shapes follow the pages' workloads: a Qwen3-class vocabulary (V = 151936),
block size 7 and Markov rank 256 ("Qwen3.8-Flash-Next DSpark 训练实验",
实验设置; "DeepSpec 训练全流程详解", 5.1 模型配置).  The value recipes are
the five workloads of the benchmark suite:

  tiny     R=1,  V=4096,  r=32,  fp32; U ~ N(0,2^2) + 6 on one uniform token
           per row; E, W ~ N(0,0.05^2); conf ~ Beta(6,2); P = U + N(0,0.5^2);
           SPS(B) = 1/(1e-3 + 2e-5 max(0, B-16)); greedy.
  greedy   R=16, V=151936, r=256, bf16; U ~ N(0,3^2) + 8 on a Zipf(1.1)-ranked
           token of one global random permutation; E, W ~ N(0,0.02^2);
           conf = Beta(6,2) * 0.9^j; P = U + N(0,0.5^2); same SPS formula.
  sampled  R=64, as greedy but P = U + N(0,1), temperature 1.
  highconc R=256, as greedy but conf ~ Beta(alpha_r, 2), alpha_r ~ U[1,10];
           SPS = 1e3 for B <= 256, 1e3 * 256 / B above, 1024 entries.
  overlap  N=4096 blocks x 7 positions, V=151936, bf16; Q ~ N(0,3^2) + Zipf
           peaks; P = Q + N(0, sigma^2), sigma ~ U[0.2, 2] per block; 15% of
           blocks have 1..6 trailing invalid positions.

  loss     B=512 blocks x 7 positions (one training sample's 512 anchors,
           "DeepSpec 训练全流程详解" 3.3 Step 1), V=151936, r=256, bf16;
           U ~ N(0,3^2) + 8 on a Zipf(1.1) token; target = that token, or a
           uniform token with probability 0.2; prev_tok = the block's anchor
           token (uniform) at j = 0 and target[j-1] after it (teacher
           forcing); P = U + N(0, sigma^2), sigma ~ U[0.2, 2] per block;
           E, W ~ N(0,0.02^2); conf_logit ~ N(0, 1.5^2).

  confidence  R requests x 7 positions, hidden size H (2560 for the pages'
           draft backbone), Markov rank r: h ~ N(0,1); w_c ~ N(0, 0.5^2 / H)
           on the hidden part and N(0, 0.5^2 / r) / 0.02 on the Markov part
           (so both halves move the logit by about 0.5); b_c = 1.2 (a mean
           confidence near 0.77); E ~ N(0, 0.02^2); prev_tok and drafted
           tokens uniform.
  gated    the gated Markov head's extra inputs for a cycle workload: hidden
           states h ~ N(0,1) [R, gamma, H]; W_g [rank, H + rank] with the
           hidden columns ~ N(0, 1/H) and the Markov columns ~ N(0, 1/rank) /
           e_std (each half moves a gate's argument by about 1).
  rnn      the RNN head's extra inputs: h as for the gated head; W_rnn
           [3, rank, 2 rank + H] (gate, candidate, output) with the state
           columns ~ N(0, 1/rank), the Markov columns ~ N(0, 1/rank) / e_std
           and the hidden columns ~ N(0, 1/H), so each block of columns moves
           an argument by about 1.
  calibration  M requests x 7 positions: predicted per-step confidence
           c ~ Beta(6,2) * 0.97^j; realised accept lengths drawn as the
           leading successes of Bernoulli(max(0, c - 0.05)) chains (a head
           that is 5 points optimistic, as in the paper-reading page's
           example).

P has gamma+1 rows per request: row gamma (the bonus row) is a fresh draw with
U's recipe plus the same noise.  Big tensors are drawn with a seeded
torch.Generator on the requested device; small ones (tokens, confidences,
per-request parameters) with numpy's default_rng(seed).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

QWEN3_VOCAB = 151936
BLOCK = 7
MARKOV_RANK = 256


@dataclass
class CycleSpec:
    name: str
    R: int
    G: int = BLOCK
    V: int = QWEN3_VOCAB
    r: int = MARKOV_RANK
    dtype: str = "bf16"            # "bf16" or "f32"
    u_std: float = 3.0
    boost: float = 8.0
    boost_kind: str = "zipf"       # "zipf" or "uniform"
    ew_std: float = 0.02
    p_noise: float = 0.5
    conf_kind: str = "beta62_decay"  # "beta62", "beta62_decay", "beta_alpha"
    sps_kind: str = "formula"      # "formula" or "flat_then_inverse"
    n_sps: int | None = None
    temperature: float = 0.0
    seed: int = 0
    extra: dict = field(default_factory=dict)


CYCLE_SPECS = {
    "tiny": CycleSpec("tiny", R=1, V=4096, r=32, dtype="f32", u_std=2.0, boost=6.0,
                      boost_kind="uniform", ew_std=0.05, p_noise=0.5,
                      conf_kind="beta62", seed=0),
    "greedy": CycleSpec("greedy", R=16, seed=1),
    "sampled": CycleSpec("sampled", R=64, p_noise=1.0, temperature=1.0, seed=2),
    "highconc": CycleSpec("highconc", R=256, conf_kind="beta_alpha",
                          sps_kind="flat_then_inverse", n_sps=1024, seed=3),
}


@dataclass
class OverlapSpec:
    name: str = "overlap"
    N: int = 4096
    G: int = BLOCK
    V: int = QWEN3_VOCAB
    q_std: float = 3.0
    boost: float = 8.0
    sigma_lo: float = 0.2
    sigma_hi: float = 2.0
    ragged_frac: float = 0.15
    seed: int = 4


@dataclass
class LossSpec:
    name: str = "loss"
    B: int = 512
    G: int = BLOCK
    V: int = QWEN3_VOCAB
    r: int = MARKOV_RANK
    u_std: float = 3.0
    boost: float = 8.0
    ew_std: float = 0.02
    sigma_lo: float = 0.2
    sigma_hi: float = 2.0
    target_noise: float = 0.2
    conf_std: float = 1.5
    seed: int = 5


def scaled(spec: CycleSpec, **kw) -> CycleSpec:
    d = dict(spec.__dict__)
    d.update(kw)
    return CycleSpec(**d)


def _torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _zipf_ranks(rng: np.random.Generator, n: int, V: int, s: float = 1.1):
    """Ranks k in 1..V with P(k) proportional to k^-s (truncated Zipf)."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1) + 1


def _boost_tokens(rng, n_rows: int, V: int, kind: str, perm: np.ndarray):
    if kind == "uniform":
        return rng.integers(0, V, size=n_rows)
    return perm[_zipf_ranks(rng, n_rows, V) - 1]


def _logit_rows(gen, rng, n_rows, V, std, boost, kind, perm, device):
    x = torch.randn((n_rows, V), generator=gen, device=device, dtype=torch.float32) * std
    if boost != 0.0:
        tok = torch.as_tensor(_boost_tokens(rng, n_rows, V, kind, perm), device=device)
        x[torch.arange(n_rows, device=device), tok] += boost
    return x


def sps_table(spec: CycleSpec) -> np.ndarray:
    """sps[B-1] = SPS(B), float32."""
    n = spec.n_sps or spec.R * (spec.G + 1)
    B = np.arange(1, n + 1, dtype=np.float64)
    if spec.sps_kind == "formula":
        s = 1.0 / (1e-3 + 2e-5 * np.maximum(0.0, B - 16.0))
    elif spec.sps_kind == "flat_then_inverse":
        s = np.where(B <= 256, 1e3, 1e3 * 256.0 / B)
    elif spec.sps_kind == "constant":
        s = np.full_like(B, 1e3)
    else:
        raise ValueError(spec.sps_kind)
    return s.astype(np.float32)


def cycle_inputs(spec: CycleSpec, device="cpu"):
    """All inputs of one draft-verify cycle, as torch tensors on ``device``.

    Keys: U [R,G,V], E [V,r], W [V,r], P [R,G+1,V] (spec.dtype); conf [R,G]
    f32; prev_tok [R] i32; req_id [R] u32 (as int64 holding 32-bit values);
    sps [n] f32; temperature, seed (python scalars)."""
    R, G, V, r = spec.R, spec.G, spec.V, spec.r
    rng = np.random.default_rng(spec.seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    dt = _torch_dtype(spec.dtype)
    perm = rng.permutation(V)

    U = _logit_rows(gen, rng, R * G, V, spec.u_std, spec.boost, spec.boost_kind, perm, device)
    U_bonus = _logit_rows(gen, rng, R, V, spec.u_std, spec.boost, spec.boost_kind, perm, device)
    U = U.to(dt).view(R, G, V)
    noise = torch.randn((R, G + 1, V), generator=gen, device=device) * spec.p_noise
    P = torch.cat([U.float(), U_bonus.to(dt).float().view(R, 1, V)], dim=1) + noise
    P = P.to(dt)
    del noise
    E = (torch.randn((V, r), generator=gen, device=device) * spec.ew_std).to(dt)
    W = (torch.randn((V, r), generator=gen, device=device) * spec.ew_std).to(dt)

    prev_tok = rng.integers(0, V, size=R).astype(np.int32)
    if spec.conf_kind == "beta62":
        conf = rng.beta(6.0, 2.0, size=(R, G))
    elif spec.conf_kind == "beta62_decay":
        conf = rng.beta(6.0, 2.0, size=(R, G)) * (0.9 ** np.arange(G))[None, :]
    elif spec.conf_kind == "beta_alpha":
        alpha = rng.uniform(1.0, 10.0, size=R)
        conf = rng.beta(alpha[:, None], 2.0, size=(R, G))
    elif spec.conf_kind == "ones":
        conf = np.ones((R, G))
    else:
        raise ValueError(spec.conf_kind)
    req_id = rng.permutation(1 << 20)[:R].astype(np.int64) + 1000

    return dict(
        U=U, E=E, W=W, P=P,
        conf=torch.as_tensor(conf.astype(np.float32), device=device),
        prev_tok=torch.as_tensor(prev_tok, device=device),
        req_id=torch.as_tensor(req_id.astype(np.int32), device=device),
        sps=torch.as_tensor(sps_table(spec), device=device),
        temperature=float(spec.temperature),
        seed=int(0x5EED0000 + spec.seed * 7919),
    )


def overlap_valid_len(spec: OverlapSpec) -> np.ndarray:
    rng = np.random.default_rng(spec.seed + 1000)
    vl = np.full(spec.N, spec.G, dtype=np.int32)
    ragged = rng.random(spec.N) < spec.ragged_frac
    vl[ragged] = spec.G - rng.integers(1, 7, size=int(ragged.sum()))
    return np.clip(vl, 0, spec.G).astype(np.int32)


def overlap_inputs(spec: OverlapSpec, device="cpu", chunk_blocks: int = 256):
    """P, Q [N,G,V] bf16, valid_len [N] i32.  Drawn chunk by chunk so the
    fp32 temporaries stay small."""
    N, G, V = spec.N, spec.G, spec.V
    rng = np.random.default_rng(spec.seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    perm = rng.permutation(V)
    sigma = rng.uniform(spec.sigma_lo, spec.sigma_hi, size=N).astype(np.float32)
    P = torch.empty((N, G, V), dtype=torch.bfloat16, device=device)
    Q = torch.empty((N, G, V), dtype=torch.bfloat16, device=device)
    for n0 in range(0, N, chunk_blocks):
        n1 = min(N, n0 + chunk_blocks)
        q = _logit_rows(gen, rng, (n1 - n0) * G, V, spec.q_std, spec.boost, "zipf",
                        perm, device).view(n1 - n0, G, V).to(torch.bfloat16)
        s = torch.as_tensor(sigma[n0:n1], device=device).view(-1, 1, 1)
        p = q.float() + torch.randn((n1 - n0, G, V), generator=gen, device=device) * s
        Q[n0:n1] = q
        P[n0:n1] = p.to(torch.bfloat16)
    vl = torch.as_tensor(overlap_valid_len(spec), device=device)
    return dict(P=P, Q=Q, valid_len=vl)


def loss_inputs(spec: LossSpec, device="cpu", chunk_blocks: int = 128):
    """U, P [B,G,V] bf16; E, W [V,r] bf16; prev_tok, target [B,G] i32;
    conf_logit [B,G] f32.  Drawn chunk by chunk so the fp32 temporaries stay
    small."""
    B, G, V, r = spec.B, spec.G, spec.V, spec.r
    rng = np.random.default_rng(spec.seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    perm = rng.permutation(V)
    sigma = rng.uniform(spec.sigma_lo, spec.sigma_hi, size=B).astype(np.float32)
    peak = _boost_tokens(rng, B * G, V, "zipf", perm).reshape(B, G)
    noisy = rng.random((B, G)) < spec.target_noise
    target = np.where(noisy, rng.integers(0, V, size=(B, G)), peak).astype(np.int32)
    prev_tok = np.empty((B, G), dtype=np.int32)
    prev_tok[:, 0] = rng.integers(0, V, size=B)
    prev_tok[:, 1:] = target[:, :-1]
    conf_logit = (rng.standard_normal((B, G)) * spec.conf_std).astype(np.float32)
    U = torch.empty((B, G, V), dtype=torch.bfloat16, device=device)
    P = torch.empty((B, G, V), dtype=torch.bfloat16, device=device)
    peak_t = torch.as_tensor(peak.reshape(-1), device=device)
    for b0 in range(0, B, chunk_blocks):
        b1 = min(B, b0 + chunk_blocks)
        n = (b1 - b0) * G
        u = torch.randn((n, V), generator=gen, device=device, dtype=torch.float32) * spec.u_std
        u[torch.arange(n, device=device), peak_t[b0 * G:b1 * G]] += spec.boost
        u = u.view(b1 - b0, G, V).to(torch.bfloat16)
        s = torch.as_tensor(sigma[b0:b1], device=device).view(-1, 1, 1)
        p = u.float() + torch.randn((b1 - b0, G, V), generator=gen, device=device) * s
        U[b0:b1] = u
        P[b0:b1] = p.to(torch.bfloat16)
    E = (torch.randn((V, r), generator=gen, device=device) * spec.ew_std).to(torch.bfloat16)
    W = (torch.randn((V, r), generator=gen, device=device) * spec.ew_std).to(torch.bfloat16)
    return dict(U=U, P=P, E=E, W=W,
                prev_tok=torch.as_tensor(prev_tok, device=device),
                target=torch.as_tensor(target, device=device),
                conf_logit=torch.as_tensor(conf_logit, device=device))


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Exact widening to a host numpy array (bf16 -> fp32 is exact)."""
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def bytes_of(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def fmt_spec(spec) -> str:
    return ", ".join(f"{k}={v}" for k, v in spec.__dict__.items() if k != "extra")


__all__ = [
    "CycleSpec", "OverlapSpec", "LossSpec", "CYCLE_SPECS", "scaled", "cycle_inputs",
    "overlap_inputs", "loss_inputs", "overlap_valid_len", "sps_table", "to_numpy", "bytes_of",
    "QWEN3_VOCAB", "BLOCK", "MARKOV_RANK",
]


def confidence_inputs(R: int, G: int, H: int, V: int, r: int, seed: int = 7,
                      dtype: str = "bf16", device="cpu"):
    """h [R,G,H], E [V,r], w_c [H+r] in dtype; b_c float; prev_tok [R],
    tokens [R,G] i32 (see the module docstring)."""
    rng = np.random.default_rng(seed)
    td = _torch_dtype(dtype)
    h = rng.standard_normal((R, G, H), dtype=np.float32)
    E = (rng.standard_normal((V, r), dtype=np.float32) * 0.02).astype(np.float32)
    w = np.concatenate([rng.standard_normal(H, dtype=np.float32) * (0.5 / np.sqrt(H)),
                        rng.standard_normal(r, dtype=np.float32) * (0.5 / np.sqrt(r) / 0.02)])
    prev_tok = rng.integers(0, V, size=R).astype(np.int32)
    tokens = rng.integers(0, V, size=(R, G)).astype(np.int32)
    to = lambda a: torch.as_tensor(a).to(device=device, dtype=td)
    return dict(h=to(h), E=to(E), w_c=to(w.astype(np.float32)), b_c=1.2,
                prev_tok=torch.as_tensor(prev_tok, device=device),
                tokens=torch.as_tensor(tokens, device=device))


def calibration_inputs(M: int, G: int, seed: int = 8, device="cpu"):
    """conf [M,G] f32 predicted per-step confidences; accept_len [M] i32
    (see the module docstring)."""
    rng = np.random.default_rng(seed)
    c = (rng.beta(6.0, 2.0, size=(M, G)) * 0.97 ** np.arange(G)).astype(np.float32)
    u = rng.random((M, G))
    ok = u < np.maximum(c.astype(np.float64) - 0.05, 0.0)
    acc = np.where(ok.all(axis=1), G, np.argmin(ok, axis=1)).astype(np.int32)
    return dict(conf=torch.as_tensor(c, device=device),
                accept_len=torch.as_tensor(acc, device=device))


def gate_inputs(R: int, G: int, H: int, r: int, e_std: float, seed: int = 9,
                dtype: str = "bf16", device="cpu"):
    """h [R,G,H] and W_g [r, H+r] in dtype (see the module docstring)."""
    rng = np.random.default_rng(seed)
    td = _torch_dtype(dtype)
    h = rng.standard_normal((R, G, H), dtype=np.float32)
    Wg = np.concatenate([rng.standard_normal((r, H), dtype=np.float32) / np.sqrt(H),
                         rng.standard_normal((r, r), dtype=np.float32) / np.sqrt(r) / e_std],
                        axis=1)
    to = lambda a: torch.as_tensor(a).to(device=device, dtype=td)
    return dict(h=to(h), W_g=to(Wg.astype(np.float32)))


def rnn_inputs(R: int, G: int, H: int, r: int, e_std: float, seed: int = 10,
               dtype: str = "bf16", device="cpu"):
    """h [R,G,H] and W_rnn [3, r, 2r+H] in dtype (see the module docstring)."""
    rng = np.random.default_rng(seed)
    td = _torch_dtype(dtype)
    h = rng.standard_normal((R, G, H), dtype=np.float32)
    Wr = np.concatenate([rng.standard_normal((3, r, r), dtype=np.float32) / np.sqrt(r),
                         rng.standard_normal((3, r, r), dtype=np.float32) / np.sqrt(r) / e_std,
                         rng.standard_normal((3, r, H), dtype=np.float32) / np.sqrt(H)],
                        axis=2)
    to = lambda a: torch.as_tensor(a).to(device=device, dtype=td)
    return dict(h=to(h), W_rnn=to(Wr.astype(np.float32)))
