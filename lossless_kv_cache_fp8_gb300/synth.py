"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers; it holds none of the codec's
arithmetic, so both the CUDA path and the CPU oracle consume the same bytes
from it.  The speculative-KV-coding page measured real Qwen3 KV caches
("early results"); those caches, models and prompts are not available, so
seeded caches with the same shapes stand in for them:

* KV caches ``[layer][k/v][kv_head][token][head_dim]``: per-channel scale
  ``sigma_c = exp(U(ln 0.1, ln 2))``, 2% of channels (chosen by the seed) 10x
  larger; ``x ~ N(0, sigma_c)``; target = cast(x); predictor =
  cast(x + eps) with ``eps ~ Laplace(0, eps_scale * sigma_c)`` (0.05 for FP8,
  0.01 for BF16).  The cast is round-to-nearest-even (torch).
* Transform-coefficient stream ``[token][coef]`` (the DCKV page's setting):
  ``b_c = exp(U(ln 0.3, ln 20))``, step ``Delta_c = exp(U(0, ln 32))``,
  mean ``mu'_{t,c} ~ N(0, (4 b_c)^2)``, ``y ~ Laplace(mu', b_c)``,
  ``q = clamp(rint(y / Delta_c), +-32767)``; the coder receives
  ``mu = mu' / Delta_c`` (fp32) and ``beta_c = b_c / Delta_c`` (fp32);
  components with ``beta_c < 0.05`` are switched off and their q set to 0.

Random draws use torch generators (a CPU generator for per-channel
parameters, the tensor's device generator for the bulk).  Bytes drawn on one
device are copied, never regenerated, when the other side needs them.
"""
from __future__ import annotations

import dataclasses
import math

import torch

FP8, BF16, COEF = 1, 2, 3
BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: int
    n_layers: int = 0
    n_kv: int = 2
    n_heads: int = 8
    head_dim: int = 128
    n_tokens: int = 0
    n_coef: int = 0
    lane_syms: int = 1024
    n_calib: int = 256
    eps_scale: float = 0.05
    index: int = 0

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index

    @property
    def elem_bytes(self) -> int:
        return 1 if self.dtype == FP8 else 2

    @property
    def n_positions(self) -> int:
        if self.dtype == COEF:
            return self.n_tokens * self.n_coef
        return self.n_layers * self.n_kv * self.n_heads * self.n_tokens * self.head_dim

    @property
    def raw_bytes(self) -> int:
        """bytes of the cache being coded (the target)"""
        return self.n_positions * self.elem_bytes

    def shape(self):
        if self.dtype == COEF:
            return (self.n_tokens, self.n_coef)
        return (self.n_layers, self.n_kv, self.n_heads, self.n_tokens, self.head_dim)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: Qwen3-0.6B / 8B / 32B KV shapes (8 KV heads, head_dim 128) and a
# hybrid model's coefficient stream (32768 tokens x 2048 coefficients).
WORKLOADS = {
    "qwen3-0.6b-1k-fp8": Workload("qwen3-0.6b-1k-fp8", FP8, n_layers=28, n_tokens=1024,
                                  lane_syms=1024, eps_scale=0.05, index=0),
    "qwen3-0.6b-8k-bf16": Workload("qwen3-0.6b-8k-bf16", BF16, n_layers=28, n_tokens=8192,
                                   lane_syms=1024, eps_scale=0.01, index=1),
    "qwen3-8b-32k-fp8": Workload("qwen3-8b-32k-fp8", FP8, n_layers=36, n_tokens=32768,
                                 lane_syms=4096, eps_scale=0.05, index=2),
    "qwen3-32b-128k-fp8": Workload("qwen3-32b-128k-fp8", FP8, n_layers=64, n_tokens=131072,
                                   lane_syms=4096, eps_scale=0.05, index=3),
    "hybrid-coef-32k-x2048": Workload("hybrid-coef-32k-x2048", COEF, n_tokens=32768, n_coef=2048,
                                      lane_syms=1024, n_calib=0, index=4),
}
WORKLOAD_ORDER = list(WORKLOADS)


def _laplace(shape, scale, gen, device):
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32) - 0.5
    a = u.abs().clamp_(max=0.5 - 2.0 ** -25)
    return -scale * torch.sign(u) * torch.log1p(-2.0 * a)


def _cast_bits(v: torch.Tensor, dtype: int) -> torch.Tensor:
    if dtype == FP8:
        return v.to(torch.float8_e4m3fn).view(torch.uint8)
    return v.to(torch.bfloat16).view(torch.int16)


def channel_sigma(w: Workload) -> torch.Tensor:
    """per-channel scale sigma_c, [layer][kv][head][head_dim] on the CPU"""
    g = torch.Generator().manual_seed(w.seed)
    shp = (w.n_layers, w.n_kv, w.n_heads, w.head_dim)
    n = math.prod(shp)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    sig = torch.exp(math.log(0.1) + u * (math.log(2.0) - math.log(0.1)))
    n_out = max(1, round(0.02 * n))
    idx = torch.randperm(n, generator=g)[:n_out]
    sig[idx] *= 10.0
    return sig.view(shp).to(torch.float32)


def gen_kv(w: Workload, device="cpu", layers=None):
    """(target_bits, pred_bits): uint8 (FP8) or int16 (BF16 bit patterns) tensors of
    shape [layer][kv][head][token][head_dim] on `device`.  `layers` restricts the
    draw to a range of layers (same values as the full draw)."""
    assert w.dtype in (FP8, BF16)
    sig = channel_sigma(w)
    lo, hi = (0, w.n_layers) if layers is None else layers
    tdt = torch.uint8 if w.dtype == FP8 else torch.int16
    shp = (hi - lo, w.n_kv, w.n_heads, w.n_tokens, w.head_dim)
    target = torch.empty(shp, dtype=tdt, device=device)
    pred = torch.empty(shp, dtype=tdt, device=device)
    for li in range(lo, hi):
        # one generator per layer so that any layer range reproduces the full draw
        g = torch.Generator(device=device).manual_seed(w.seed * 1000003 + li)
        s = sig[li].to(device).view(w.n_kv, w.n_heads, 1, w.head_dim)
        x = torch.randn((w.n_kv, w.n_heads, w.n_tokens, w.head_dim), generator=g,
                        device=device, dtype=torch.float32) * s
        eps = _laplace(x.shape, w.eps_scale * s, g, device)
        target[li - lo] = _cast_bits(x, w.dtype)
        pred[li - lo] = _cast_bits(x + eps, w.dtype)
        del x, eps
    return target, pred


def gen_coef(w: Workload, device="cpu"):
    """(q int16 [T][C], mu fp32 [T][C], beta fp32 [C]) on `device`."""
    assert w.dtype == COEF
    g = torch.Generator().manual_seed(w.seed)
    C = w.n_coef
    b = torch.exp(math.log(0.3) + torch.rand(C, generator=g, dtype=torch.float64)
                  * (math.log(20.0) - math.log(0.3))).to(torch.float32)
    delta = torch.exp(torch.rand(C, generator=g, dtype=torch.float64) * math.log(32.0)).to(torch.float32)
    beta = b / delta
    gd = torch.Generator(device=device).manual_seed(w.seed * 1000003 + 7)
    bd, dd = b.to(device), delta.to(device)
    mu_y = torch.randn((w.n_tokens, C), generator=gd, device=device, dtype=torch.float32) * (4.0 * bd)
    y = mu_y + _laplace(mu_y.shape, bd, gd, device)
    q = torch.round(y / dd).clamp_(-32767, 32767).to(torch.int16)
    mu = (mu_y / dd).to(torch.float32)
    off = ~(beta >= 0.05)
    q[:, off.to(device)] = 0
    return q, mu, beta.to(device)


def gen_workload(w: Workload, device="cpu"):
    """Uniform entry: returns (target, pred, calib_pred) where calib_pred is the
    second input of calibration (the predictor cache for KV, beta for COEF) and
    pred is the second input of encode/decode (the predictor cache, or mu)."""
    if w.dtype == COEF:
        q, mu, beta = gen_coef(w, device)
        return q, mu, beta
    t, p = gen_kv(w, device)
    return t, p, p


def to_paged(target, pred, block_tokens: int, spare_blocks: int = 3, seed: int = 0):
    """Copies dense caches [layer][kv][head][token][head_dim] into paged pools
    [layer][kv][n_blocks][block_tokens][head][head_dim] under a seeded random
    block table: the token blocks go to a random permutation of the pool's
    blocks, `spare_blocks` blocks stay unused, and rows past the last token are
    zero.  Returns (target_pool, pred_pool, block_table (int32 holding u32
    block indices), n_blocks)."""
    L, KV, H, T, D = target.shape
    B = block_tokens
    ntb = -(-T // B)
    n_blocks = ntb + spare_blocks
    g = torch.Generator().manual_seed(BASE_SEED * 7 + seed)
    perm = torch.randperm(n_blocks, generator=g)[:ntb]

    def pack(x):
        xt = x.permute(0, 1, 3, 2, 4)                     # [L][kv][T][H][D]
        pad = ntb * B - T
        if pad:
            xt = torch.cat([xt, torch.zeros((L, KV, pad, H, D), dtype=x.dtype, device=x.device)], dim=2)
        pool = torch.zeros((L, KV, n_blocks, B, H, D), dtype=x.dtype, device=x.device)
        pool[:, :, perm.to(x.device)] = xt.reshape(L, KV, ntb, B, H, D)
        return pool

    return pack(target), pack(pred), perm.to(torch.int32).to(target.device), n_blocks


# ---- checkerboard context (the DCKV page's two-pass context model) --------------------------
# The page's learned rank-1024 map is replaced by a seeded one: two integer factor
# matrices with entries in [-8, 8].  The generator below uses them as a real-valued
# linear map (no quantisation), so the coded data carries the structure a context
# model can exploit; the coder's own integer arithmetic is not part of this module.
CTX_RANK, CTX_SHIFT1, CTX_SHIFT2 = 1024, 6, 8


def ctx_map(n_coef: int, rank: int = CTX_RANK, seed: int = 0):
    """(V int8 [rank][n_coef], U int8 [n_coef][rank]), entries uniform in [-8, 8]"""
    g = torch.Generator().manual_seed(BASE_SEED * 13 + seed)
    V = torch.randint(-8, 9, (rank, n_coef), generator=g, dtype=torch.int32).to(torch.int8)
    U = torch.randint(-8, 9, (n_coef, rank), generator=g, dtype=torch.int32).to(torch.int8)
    return V, U


def gen_coef_checkerboard(w: Workload, device="cpu", rank: int = CTX_RANK):
    """Coefficient rows split by token parity.  Even rows are gen_coef's rows.
    Odd row t (token 2t + 1) has mean mu_t + U V x_t / 2^(s1 + s2) / 16 (step
    units), x_t = clamp(q_{2t} + q_{2t+2}, +-127) (a missing right neighbour is
    0), and q = clamp(rint(mean + Laplace(0, beta_c)), +-32767) (switched-off
    components 0).  Returns (q_even, q_odd, mu_even, mu_odd, beta, V, U)."""
    assert w.dtype == COEF
    q, mu, beta = gen_coef(w, device)
    T, C = q.shape
    V, U = ctx_map(C, rank)
    q_even, mu_even, mu_odd = q[0::2].contiguous(), mu[0::2].contiguous(), mu[1::2].contiguous()
    T_o = T // 2
    right = torch.zeros((T_o, C), dtype=torch.int64, device=device)
    n_r = min(T_o, q_even.shape[0] - 1)
    right[:n_r] = q_even[1:1 + n_r].to(torch.int64)
    x = (q_even[:T_o].to(torch.int64) + right).clamp_(-127, 127).to(torch.float64)
    shift = (x @ V.to(device).to(torch.float64).T) @ U.to(device).to(torch.float64).T
    shift = shift / float(1 << (CTX_SHIFT1 + CTX_SHIFT2)) / 16.0
    gd = torch.Generator(device=device).manual_seed(w.seed * 1000003 + 11)
    bd = beta.to(device)
    noise = _laplace((T_o, C), bd, gd, device).to(torch.float64)
    q_odd = torch.round(mu_odd.to(torch.float64) + shift + noise).clamp_(-32767, 32767).to(torch.int16)
    q_odd[:, ~(beta >= 0.05).to(device)] = 0
    return q_even, q_odd, mu_even, mu_odd, beta.to(device), V.to(device), U.to(device)
